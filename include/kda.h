/*
 * kda.h: C ABI of the GB300 (sm_103a) Kimi Delta Attention library, libkda.so.
 *
 * The library computes the KDA recurrence, i.e. the gated delta rule with one
 * decay per key channel, over a pool of fp32 states.  For one (sequence, value
 * head) with state S (dv x dk, "V x K": rows are value channels) and one token
 * (q, k in R^dk, v in R^dv, g in R^dk, scalar b):
 *
 *   q^ = q / sqrt(sum q^2 + eps),  k^ = k / sqrt(sum k^2 + eps)   (Q/K L2Norm)
 *   alpha_c = exp(g_c),  beta = sigmoid(b)            (gate and beta processing)
 *   S' = S diag(alpha)                                (state decay)
 *   u  = beta (v - S' k^)                             (delta rule)
 *   S  = S' + u k^T                                   (outer-product update)
 *   o  = scale * S q^                                 (output)
 *   and S is written back in place                    (final-state write-back)
 *
 * Source of the step list: "Ascend day-0 support for Kimi K3"
 * (hwcomputing.csdn.net/6a695b59...), section "Fused-operator acceleration:
 * KDA Prefill and Decode dual path" (decode kernel paragraph; prefill in
 * 64-token chunks; decode/MTP updates run directly on the state pool).
 * Speculative verify/commit: "2.8x faster Kimi K3 inference on CANN"
 * (hwcomputing.csdn.net/6ac7907e...), section 04 "ReplaySSM".
 *
 * Conventions shared by every entry point
 * ----------------------------------------
 * - All tensor pointers are DEVICE pointers to contiguous row-major buffers,
 *   16-byte aligned.  The caller allocates and frees everything; the library
 *   never allocates device memory.  Every entry point but one keeps no global
 *   mutable state, so calls on different streams are independent (given
 *   separate outputs and workspaces).  The exception is
 *   kda_prefill_chunked_static, whose scratch is one device array shared by
 *   all its calls; see its comment below.
 * - State pool: float32 [num_slots][H][dv][dk]; the state of (slot, head) is
 *   one contiguous dv x dk block with dk fastest.
 * - Slot ids are int32.  A negative slot id marks a padding entry: it is
 *   skipped (outputs zero, no state access, no error).  A slot id >= num_slots
 *   is an error: that entry is skipped the same way and KDA_DEVERR_SLOT is
 *   OR-ed into *err_flag (when err_flag is non-NULL).  The same slot id twice
 *   in one call is a precondition violation (the result is unspecified).
 * - dtype: q, k, v, b and outputs share one element type (kda_dtype); g is
 *   always float32; states and update records are float32.
 * - Supported head sizes: dk and dv each in {32, 64, 128}.
 * - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *   default stream) and never synchronise the host.  A host-detectable
 *   argument error returns a negative kda_status and launches nothing.
 *   A batch of 0 (or 0 tokens) returns KDA_OK and launches nothing.
 * - Results are deterministic: no atomics touch data, so the same inputs give
 *   bit-identical outputs and states run to run and regardless of batch order.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KDA_ABI_VERSION 6

#if defined(__GNUC__)
#define KDA_API __attribute__((visibility("default")))
#else
#define KDA_API
#endif

typedef enum kda_status {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = -1,  /* NULL pointer, negative size, misalignment,
                                  draft length outside 1..16, bad dims        */
    KDA_ERR_UNSUPPORTED = -2,  /* dk/dv/dtype combination not built           */
    KDA_ERR_CUDA = -3,         /* a CUDA runtime call or launch failed        */
    KDA_ERR_WORKSPACE = -4     /* workspace NULL, too small or unaligned     */
} kda_status;

typedef enum kda_dtype {
    KDA_DT_F32 = 0,
    KDA_DT_BF16 = 1
} kda_dtype;

/* Bits OR-ed into *err_flag by the kernels (device-detected errors). */
enum {
    KDA_DEVERR_SLOT = 1,      /* slot id >= num_slots                          */
    KDA_DEVERR_ACCEPTED = 2,  /* num_accepted outside 0..draft_len             */
    KDA_DEVERR_SEQLENS = 4,   /* cu_seqlens not non-decreasing / past total_T  */
    KDA_DEVERR_TIMEOUT = 8,   /* an internal bounded wait gave up (prefill)    */
    KDA_DEVERR_RANGE = 16,    /* a value passed to the tensor-core prefill's
                                 fp16 products exceeded +-65504; the outputs and
                                 final state of that sequence are not valid  */
    KDA_DEVERR_SNAPSHOT = 32, /* a prefill snapshot request was skipped: token
                                 count not a positive multiple of 64 within its
                                 sequence, requests out of order, or slot id
                                 >= num_slots                                */
    KDA_DEVERR_BOUNDS = 64,   /* (checked builds, -DKDA_CHECKED, only) an
                                 access outside its buffer was found and
                                 skipped                                     */
    KDA_DEVERR_DUPLICATE = 128 /* (checked builds only) a slot id appears
                                 twice in one call's slot_ids (the call's
                                 results for those slots are not valid)      */
};

typedef struct kda_dims {
    int32_t num_heads;  /* H >= 1; q, k, v share the head count               */
    int32_t dk;         /* key head size, in {32, 64, 128}                    */
    int32_t dv;         /* value head size, in {32, 64, 128}                  */
    int32_t dtype;      /* kda_dtype of q, k, v, b and of the outputs         */
    float eps;          /* L2Norm epsilon inside the sqrt (1e-6 typical), >=0 */
    float scale;        /* output scale; <= 0 selects dk^-1/2                 */
} kda_dims;

/*
 * ReplaySSM update records written by kda_verify_record and consumed by
 * kda_replay_commit, one per (sequence, draft token, head):
 *   k_hat  float32 [B][D][H][dk]  normalised key actually used
 *   v      dtype   [B][D][H][dv]  value (bit copy of the input)
 *   g      float32 [B][D][H][dk]  raw log-decay (bit copy of the input)
 *   beta   float32 [B][D][H]      sigmoid(b) actually used
 * Replaying record j applies exactly the arithmetic the decode kernel applies
 * for that token, so replaying a records equals a kda_decode calls bit for bit.
 */
typedef struct kda_records {
    float *k_hat;
    void *v;
    float *g;
    float *beta;
} kda_records;

/*
 * kda_decode: one token for each of `batch` sequences, fused single launch.
 * Computes every step listed at the top for token n on the state of
 * (slot_ids[n], h), for all heads h, and writes the state back in place.
 * (Decode kernel paragraph of the "KDA Prefill and Decode dual path" section:
 * one work item per logical sequence x value head.)
 *
 *   q, k     dtype  [batch][H][dk]
 *   v        dtype  [batch][H][dv]
 *   g        f32    [batch][H][dk]
 *   b        dtype  [batch][H]
 *   slot_ids i32    [batch]
 *   pool     f32    [num_slots][H][dv][dk]   read and written in place
 *   out      dtype  [batch][H][dv]           written (zero for skipped entries)
 *   err_flag i32*   optional device word, device errors OR-ed in
 */
KDA_API int kda_decode(const kda_dims *dims, int32_t batch, const void *q,
               const void *k, const void *v, const float *g, const void *b,
               const int32_t *slot_ids, float *pool, int64_t num_slots,
               void *out, int32_t *err_flag, void *stream);

/*
 * Inputs of kda_decode_fused besides the token's q, k, v, g, b:
 *   conv_state  dtype [num_slots][H][3][2 dk + dv]  the last three RAW inputs
 *               of each (slot, head), oldest first, channels ordered q | k | v;
 *               read and shifted in place (same slots as the state pool)
 *   conv_w      f32   [H][2 dk + dv][4]  depthwise conv taps per channel; tap 0
 *               multiplies the oldest input, tap 3 the current one
 *   z           dtype [batch][H][dv]     output-gate pre-activation
 *   norm_w      f32   [dv]               RMS-norm weight (shared by the heads)
 *   eps_o       RMS-norm epsilon inside the sqrt, >= 0
 * All arrays are owned by the caller.
 */
typedef struct kda_fused_io {
    void *conv_state;
    const float *conv_w;
    const void *z;
    const float *norm_w;
    float eps_o;
} kda_fused_io;

/*
 * kda_decode_fused: one MegaKDA-style fused decode step ("2.8x faster Kimi K3
 * inference on CANN", section 03 "MegaKDA": ShortConv and the output-side
 * compute fused with the KDA recurrence in one operator).  For every
 * (sequence n, head h), in one launch:
 *   x~_c = silu(w_c0 x_{t-3,c} + w_c1 x_{t-2,c} + w_c2 x_{t-1,c} + w_c3 x_c)
 *          for each channel c of q, k and v, with x_{t-3..t-1} from conv_state,
 *          which is then shifted to hold x_{t-2}, x_{t-1}, x (raw inputs)
 *   o    = the kda_decode step on (q~, k~, v~, g, b), held in fp32 (the
 *          convolved values are never rounded to dtype), state written back
 *   out  = o / sqrt(mean_i o_i^2 + eps_o) * norm_w * sigmoid(z)
 * The input projections are not part of it.  Arguments as for kda_decode,
 * plus `io`; supported shapes as for kda_decode.  Padding and out-of-range
 * slots leave the state pool and the conv state untouched and output zero.
 */
KDA_API int kda_decode_fused(const kda_dims *dims, int32_t batch, const void *q,
               const void *k, const void *v, const float *g, const void *b,
               const int32_t *slot_ids, float *pool, int64_t num_slots,
               const kda_fused_io *io, void *out, int32_t *err_flag, void *stream);

/*
 * kda_verify_record: ReplaySSM verification of `draft_len` (1..16) draft
 * tokens per sequence.  Evaluates the recurrence over the draft tokens,
 * starting from the committed state of (slot_ids[n], h), WITHOUT writing the
 * pool; emits the output of every draft token and stores only the update
 * records (kda_records) instead of per-token states ("2.8x faster Kimi K3
 * inference on CANN", section 04 "ReplaySSM").  The outputs are computed
 * from the window's chunk form, so they equal those of draft_len sequential
 * kda_decode calls up to rounding (not bit for bit); the records are the
 * decode routine's own coefficients, so committing them reproduces decode
 * bit for bit.
 *
 *   q, k     dtype  [batch][draft_len][H][dk]
 *   v        dtype  [batch][draft_len][H][dv]
 *   g        f32    [batch][draft_len][H][dk]
 *   b        dtype  [batch][draft_len][H]
 *   pool     f32    [num_slots][H][dv][dk]   read only
 *   out      dtype  [batch][draft_len][H][dv]
 *   rec      records sized for (batch, draft_len); all four arrays written
 *            for every entry, padding and errors included (they only depend
 *            on the token inputs).
 *   workspace      device scratch of at least
 *                  kda_verify_workspace_bytes(dims, batch, draft_len) bytes,
 *                  256-byte aligned, owned by the caller; it may be NULL
 *                  when that size is 0.  Its contents on return are
 *                  undefined.  Calls sharing one workspace must not overlap
 *                  on the GPU.  A required workspace that is NULL, too small
 *                  or unaligned returns KDA_ERR_WORKSPACE, launching nothing.
 */
KDA_API int kda_verify_record(const kda_dims *dims, int32_t batch, int32_t draft_len,
                      const void *q, const void *k, const void *v,
                      const float *g, const void *b, const int32_t *slot_ids,
                      const float *pool, int64_t num_slots, void *out,
                      const kda_records *rec, void *workspace,
                      size_t workspace_bytes, int32_t *err_flag, void *stream);

/*
 * Workspace bytes kda_verify_record needs for (dims, batch, draft_len): about
 * 12.6 KB per (sequence, head) for bf16 windows of up to 8 tokens at
 * dk = dv = 128 (the per-(sequence, head) window products and the decayed key
 * and query tile the state kernel consumes), 0 for every other shape.  0 for
 * invalid arguments.
 */
KDA_API size_t kda_verify_workspace_bytes(const kda_dims *dims, int32_t batch,
                                          int32_t draft_len);

/*
 * kda_replay_commit: commit after acceptance.  For each sequence n with
 * a = num_accepted[n] (0..draft_len), replays records 0..a-1 in order onto
 * the committed state of (slot_ids[n], h) and writes it back:
 *   S = S diag(exp g_j);  S = S + beta_j (v_j - S k_hat_j) k_hat_j^T.
 * a == 0 leaves the state untouched (no memory access).  a outside
 * 0..draft_len sets KDA_DEVERR_ACCEPTED and skips the sequence.
 *
 *   rec          records written by kda_verify_record for the same
 *                (batch, draft_len, dims)
 *   num_accepted i32 [batch] device
 *   slot_ids     i32 [batch] device (normally those given to verify)
 *   pool         f32 [num_slots][H][dv][dk] read and written in place
 */
KDA_API int kda_replay_commit(const kda_dims *dims, int32_t batch, int32_t draft_len,
                      const kda_records *rec, const int32_t *num_accepted,
                      const int32_t *slot_ids, float *pool, int64_t num_slots,
                      int32_t *err_flag, void *stream);

/*
 * ReplaySSM variant records ("2.8x faster Kimi K3 inference on CANN", section
 * 04 "ReplaySSM": during verification only per-token update records are
 * kept).  Here the record of (sequence n, draft token j, head h) holds the
 * update itself instead of the value:
 *   k_hat  float32 [B][D][H][dk]  normalised key
 *   g      float32 [B][D][H][dk]  raw log-decay (bit copy of the input)
 *   u      float32 [B][D][H][dv]  u_j = beta_j (v_j - S'_j k^_j), the delta
 *                                 rule's correction along k^_j, where S'_j is
 *                                 the decayed state before token j
 * so that committing token j is S <- S diag(exp g_j) + u_j k^_j^T: no dot
 * product, one multiply and one fused multiply-add per state element.  u
 * comes from verify's window form, so a u-record commit equals a decode
 * sequence up to rounding (not bit for bit; the value-record commit of
 * kda_replay_commit keeps that contract).  A u-record commit and the fused
 * commit of kda_commit_verify_u give the same bits.  1536 bytes per
 * token-head at dk = dv = 128 (against 1284 for kda_records).
 */
typedef struct kda_records_u {
    float *k_hat;
    float *g;
    float *u;
} kda_records_u;

/* Total bytes of the three u-record arrays for (batch, draft_len). */
KDA_API size_t kda_records_u_bytes(const kda_dims *dims, int32_t batch, int32_t draft_len);

/*
 * kda_verify_record_u: kda_verify_record writing u records.  Arguments,
 * workspace and outputs as kda_verify_record (the outputs are the same
 * bits); rec->u of a padding or out-of-range entry is zero.
 */
KDA_API int kda_verify_record_u(const kda_dims *dims, int32_t batch, int32_t draft_len,
                                const void *q, const void *k, const void *v,
                                const float *g, const void *b, const int32_t *slot_ids,
                                const float *pool, int64_t num_slots, void *out,
                                const kda_records_u *rec, void *workspace,
                                size_t workspace_bytes, int32_t *err_flag, void *stream);

/*
 * kda_replay_commit_u: commit from u records.  For each sequence n with
 * a = num_accepted[n] (0..draft_len), applies records 0..a-1 in order:
 * S = S diag(exp g_j) + u_j k_hat_j^T, and writes the state back.  a == 0
 * leaves it untouched; a outside 0..draft_len sets KDA_DEVERR_ACCEPTED.
 * The pool must hold the state verify read (precondition).
 */
KDA_API int kda_replay_commit_u(const kda_dims *dims, int32_t batch, int32_t draft_len,
                                const kda_records_u *rec, const int32_t *num_accepted,
                                const int32_t *slot_ids, float *pool, int64_t num_slots,
                                int32_t *err_flag, void *stream);

/*
 * kda_commit_verify_u: the previous window's commit and this window's
 * verify in one call, for when the previous window's acceptance is already
 * on the device (no host round trip between them).  It applies the
 * accepted prefix (prev_accepted[n] records, 0..prev_draft_len) of the
 * previous window's u records `prev` exactly as kda_replay_commit_u does
 * (same bits), writes the committed state back to the pool, and verifies
 * the new draft window from it into `rec` (as kda_verify_record_u).  On the
 * tensor-core verify shape (bf16, dk = dv = 128, draft_len <= 8, with a
 * workspace) the commit and the verify are two launches in stream order
 * (measured faster than one launch doing both); on the other shapes the
 * verify kernel commits the state it has loaded, one state read and one
 * write in one launch.  prev and rec must not overlap.  prev_accepted
 * outside 0..prev_draft_len sets KDA_DEVERR_ACCEPTED and that sequence is
 * verified without a commit.
 */
KDA_API int kda_commit_verify_u(const kda_dims *dims, int32_t batch, int32_t prev_draft_len,
                                const kda_records_u *prev, const int32_t *prev_accepted,
                                int32_t draft_len, const void *q, const void *k, const void *v,
                                const float *g, const void *b, const int32_t *slot_ids,
                                float *pool, int64_t num_slots, void *out,
                                const kda_records_u *rec, void *workspace,
                                size_t workspace_bytes, int32_t *err_flag, void *stream);

/*
 * kda_prefill_chunked: chunked prefill of a variable-length batch.
 * Sequence s covers tokens cu_seqlens[s] .. cu_seqlens[s+1]-1 of the packed
 * token axis.  The tokens are processed in 64-token chunks (the last chunk of
 * a sequence may be partial); within a chunk the work is put in WY/UT form:
 *   gamma = in-chunk cumulative sum of g (gate accumulation),
 *   T = (I + A)^-1 for the strictly lower-triangular beta-scaled decayed key
 *   Gram matrix A, W = T diag(beta) K~, U' = T diag(beta) V, and across chunks
 *   U = U' - W S^T,  O = scale (Q~ S^T + P U),  S <- S diag(e^gamma_C) + U^T K^.
 * ("KDA Prefill and Decode dual path": prefill takes 64-token chunks and
 * organises Q/K normalisation, gate accumulation and chunk KDA as batched
 * computation.)  The result equals the token-by-token recurrence up to
 * rounding.
 *
 *   cu_seqlens     i32 [num_seqs+1] device, non-decreasing, cu[0] = 0,
 *                  cu[num_seqs] <= total_tokens
 *   q, k           dtype [total_tokens][H][dk]
 *   v              dtype [total_tokens][H][dv]
 *   g              f32   [total_tokens][H][dk]
 *   b              dtype [total_tokens][H]
 *   slot_ids       i32   [num_seqs] device; the final state of sequence s is
 *                  written to slot slot_ids[s]
 *   init_from_pool 0: start from a zero state; 1: start from the slot's state
 *   out            dtype [total_tokens][H][dv]
 *   workspace      device scratch of at least
 *                  kda_prefill_workspace_bytes(dims, num_seqs, total_tokens)
 *                  bytes, 256-byte aligned, owned by the caller; its contents
 *                  on entry do not matter and are undefined on return.
 *                  Calls sharing one workspace must not overlap on the GPU.
 */
KDA_API int kda_prefill_chunked(const kda_dims *dims, int32_t num_seqs,
                        const int32_t *cu_seqlens, int64_t total_tokens,
                        const void *q, const void *k, const void *v,
                        const float *g, const void *b,
                        const int32_t *slot_ids, float *pool,
                        int64_t num_slots, int32_t init_from_pool, void *out,
                        void *workspace, size_t workspace_bytes,
                        int32_t *err_flag, void *stream);

/*
 * kda_prefill_chunked_snapshots: kda_prefill_chunked that also writes the
 * state reached at chosen chunk boundaries into pool slots, so that a later
 * prefill can resume from a cached prefix with init_from_pool = 1 (the KDA
 * Prefix-Cache of "Ascend day-0 support for Kimi K3", Kimi K3 overview; the
 * serving engine's prefix cache and chunked prefill in the vLLM Ascend
 * paragraph of the same page).  Arguments and results are those of
 * kda_prefill_chunked, plus num_snaps requests, sorted by sequence and then
 * by token count:
 *   snap_seq     i32 [num_snaps] device: the sequence (0 .. num_seqs-1)
 *   snap_tokens  i32 [num_snaps] device: t, a positive multiple of 64 with
 *                t <= that sequence's length; the snapshot is the state after
 *                the sequence's first t tokens (starting from its initial
 *                state, zero or the pool's per init_from_pool)
 *   snap_slot    i32 [num_snaps] device: destination slot; the state of every
 *                head goes to pool[snap_slot][h] (dv x dk fp32).  A negative
 *                slot skips the request silently.
 * A request that cannot be met (token count not a positive multiple of 64,
 * beyond the sequence, out of order, or slot >= num_slots) is skipped and
 * sets KDA_DEVERR_SNAPSHOT.  Requests of a padding or out-of-range sequence
 * are ignored.  Destination slots must differ from each other and from the
 * sequences' own slots (precondition).  num_snaps = 0 is kda_prefill_chunked;
 * num_snaps < 0, or a NULL request array when num_snaps > 0, returns
 * KDA_ERR_INVALID_ARG.  Each snapshot adds dv x dk x 4 bytes per head of
 * writes; the workspace is the same as kda_prefill_chunked's.
 */
KDA_API int kda_prefill_chunked_snapshots(const kda_dims *dims, int32_t num_seqs,
                                          const int32_t *cu_seqlens, int64_t total_tokens,
                                          const void *q, const void *k, const void *v,
                                          const float *g, const void *b,
                                          const int32_t *slot_ids, float *pool,
                                          int64_t num_slots, int32_t init_from_pool, void *out,
                                          int32_t num_snaps, const int32_t *snap_seq,
                                          const int32_t *snap_tokens, const int32_t *snap_slot,
                                          void *workspace, size_t workspace_bytes,
                                          int32_t *err_flag, void *stream);

/*
 * kda_prefill_fused: the MegaKDA-style fused prefill ("2.8x faster Kimi K3
 * inference on CANN", section 03 "MegaKDA"), the prefill counterpart of
 * kda_decode_fused.  For each sequence and head:
 *   - the ShortConv of kda_decode_fused runs along the sequence: the three
 *     inputs before its first token are the slot's conv state when
 *     init_from_pool is set, else zero; the convolved k and q are rounded to
 *     dtype (bf16), the convolved v stays fp32;
 *   - the chunked prefill of kda_prefill_chunked runs on the convolved
 *     inputs (init_from_pool selects the KDA state's start as there);
 *   - out = o / sqrt(mean_i o_i^2 + eps_o) * norm_w * sigmoid(z) per token;
 *   - the slot's conv state afterwards holds the last three raw inputs of the
 *     history followed by the sequence (so a decode continues from it).
 * Arguments as for kda_prefill_chunked, plus `io` (kda_fused_io, with z of
 * shape dtype [total_tokens][H][dv]).  Only the tensor-core shape (bf16,
 * dk = dv = 128) is built; every other shape returns KDA_ERR_UNSUPPORTED.
 * Padding and out-of-range sequences output zero and leave both pools alone.
 */
KDA_API int kda_prefill_fused(const kda_dims *dims, int32_t num_seqs,
                      const int32_t *cu_seqlens, int64_t total_tokens,
                      const void *q, const void *k, const void *v, const float *g,
                      const void *b, const int32_t *slot_ids, float *pool,
                      int64_t num_slots, int32_t init_from_pool,
                      const kda_fused_io *io, void *out, void *workspace,
                      size_t workspace_bytes, int32_t *err_flag, void *stream);

/*
 * kda_prefill_chunked_static: kda_prefill_chunked without a caller-provided
 * workspace, for callers that cannot allocate device memory at the point of
 * the call: code that runs while a CUDA graph is being captured (where
 * cudaMalloc is not allowed), serving engines whose device memory is planned
 * up front and owned by another allocator, and plug-in hosts that hand the
 * library only its inputs and outputs.  (The source pages have no
 * counterpart; this is an interface convenience of this library.)
 *
 * The scratch is a fixed device array inside the library of
 * KDA_STATIC_SCRATCH_BYTES bytes, reserved on every GPU that loads the
 * library until the process exits.  Arguments and results are exactly those
 * of kda_prefill_chunked, minus workspace/workspace_bytes.
 *   - Returns KDA_ERR_WORKSPACE, launching nothing, when
 *     kda_prefill_workspace_bytes(dims, num_seqs, total_tokens) exceeds
 *     KDA_STATIC_SCRATCH_BYTES (about 440 (chunk, head) pairs at
 *     dk = dv = 128 bf16; split larger batches into several calls).
 *   - Calls no allocating routine (no cudaMalloc/cudaFree).
 *   - The first call on a device looks up the array's device address on that
 *     device (cudaGetSymbolAddress); make that first call before any stream
 *     capture.  It returns KDA_ERR_CUDA if the lookup fails.
 *   - Every call on a device shares the one array, which keeps the previous
 *     call's bytes; nothing in it needs to start at zero.  Calls that overlap
 *     on the GPU (different streams, or different host threads) race on it:
 *     order them, or use kda_prefill_chunked with separate workspaces.
 */
#define KDA_STATIC_SCRATCH_BYTES ((size_t)64 << 20)

KDA_API int kda_prefill_chunked_static(const kda_dims *dims, int32_t num_seqs,
                                       const int32_t *cu_seqlens, int64_t total_tokens,
                                       const void *q, const void *k, const void *v,
                                       const float *g, const void *b,
                                       const int32_t *slot_ids, float *pool,
                                       int64_t num_slots, int32_t init_from_pool,
                                       void *out, int32_t *err_flag, void *stream);

/* KDA_STATIC_SCRATCH_BYTES of the built library. */
KDA_API size_t kda_static_scratch_bytes(void);

/* Workspace bytes kda_prefill_chunked needs for this shape (0 on bad dims). */
KDA_API size_t kda_prefill_workspace_bytes(const kda_dims *dims, int32_t num_seqs,
                                   int64_t total_tokens);

/* Total bytes of the four record arrays for (batch, draft_len). */
KDA_API size_t kda_records_bytes(const kda_dims *dims, int32_t batch,
                         int32_t draft_len);

/* Static description of a status code ("ok", "invalid argument", ...). */
KDA_API const char *kda_status_string(int status);

/* KDA_ABI_VERSION of the built library. */
KDA_API int kda_abi_version(void);

/* 1 when the library was built with its kernels' bounds checks
 * (-DKDA_CHECKED: an access outside its buffer sets KDA_DEVERR_BOUNDS in the
 * call's err_flag and is skipped), else 0. */
KDA_API int kda_checked_build(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
