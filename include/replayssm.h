/*
 * replayssm.h -- C ABI of the ReplaySSM batched decode library (sm_103a).
 *
 * The method (described on "ReplaySSM: o ganho aparece na carga concorrente,
 * não no nome da otimização", introduction, and "NVIDIA y Princeton aceleran
 * modelos híbridos al guardar entradas recientes en lugar del estado
 * completo", paragraphs 2-4): each sequence's SSM-layer state is kept as an
 * FP32 checkpoint S_c, an optional BF16 read copy of it, and a ring of the
 * last W token inputs. A decode step appends the token to the ring and
 * computes the output from the checkpoint plus the buffered inputs, writing
 * no state; the checkpoint is only rewritten when the ring fills
 * (consolidate). Speculative drafts are verified from one read of S_c and
 * accepted by moving a per-sequence pointer. The layer types are those named
 * on "NVIDIA présente ReplaySSM : accélérer le décodage des modèles hybrides
 * Mamba et GDN", section "Pourquoi les hybrides sont devenus la norme":
 * Mamba-2, Gated DeltaNet (GDN) and a Kimi-Delta-Attention-style
 * per-channel gate (KDA).
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller, dense
 *    (row-major, no padding) in the layouts stated below, and 16-byte
 *    aligned. The library never allocates, frees or synchronises.
 *  - Every call is asynchronous on `stream` (a cudaStream_t passed as void*;
 *    NULL means the legacy default stream) and returns a replayssm_status.
 *    Argument errors are detected on the host before any CUDA call and
 *    nothing is launched; REPLAYSSM_ERR_CUDA reports a launch error.
 *  - Data-dependent precondition failures (for example a full ring) are
 *    reported per sequence on the device by OR-ing bits into state->status;
 *    the affected sequence is left untouched and the others proceed. Kernels
 *    never trap and every wait they make is bounded (about one second), after
 *    which they set REPLAYSSM_SEQ_TIMEOUT and skip the remaining work.
 *  - Calls on one layer state must be ordered (one stream, or events);
 *    calls that overlap on the GPU race.
 *
 * Layouts (b = batch, H = heads, G = Mamba-2 B/C groups, W = window):
 *  Mamba-2 state    S_ckpt f32 [b, H, P, N] (N contiguous); S_read bf16 same
 *  delta state      S_ckpt f32 [b, H, d_v, d_k] (d_k contiguous); S_read same
 *  Mamba-2 token    x [b, H, P], B [b, G, N], C [b, G, N] (in_dtype);
 *                   dt [b, H] f32 (already activated, > 0)
 *  delta token      q, k [b, H, d_k], v [b, H, d_v] (in_dtype);
 *                   alpha f32 [b, H] (GDN) or [b, H, d_k] (KDA); beta f32 [b, H]
 *  ring fields      per head, slot-major inside the head so that a head's W
 *                   entries are contiguous: x [b, H, W, P]; q, k [b, H, W, d_k];
 *                   v [b, H, W, d_v]; KDA alpha [b, H, W, d_k]. Scalar fields
 *                   (dt, beta, GDN alpha) are [b, H, Wd] with Wd = W rounded up
 *                   to a multiple of 4 (pad entries unused). Mamba-2 B and C are
 *                   per group: [b, W, G, N]. Slot s of a sequence holds entry
 *                   (s - head) mod W after its checkpoint.
 *  pointers         ring_head, ring_len, status, sync: int32 [b]
 *  outputs          f32: y [b, H, P]; o [b, H, d_v]; verify o [b, K, H, d_v]
 *
 * Supported sizes (else REPLAYSSM_ERR_UNSUPPORTED): N or d_k in {64, 128};
 * P or d_v a multiple of 32 in [32, 256]; 1 <= W <= 64; heads >= 1;
 * groups divides heads; 1 <= K <= 8 and K <= W. batch == 0 is a no-op.
 */
#ifndef REPLAYSSM_H
#define REPLAYSSM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define REPLAYSSM_API __attribute__((visibility("default")))

typedef int32_t replayssm_status;

/* Host-side return codes. */
#define REPLAYSSM_OK 0
#define REPLAYSSM_ERR_INVALID_ARG 1 /* null pointer, non-positive size, bad flag */
#define REPLAYSSM_ERR_UNSUPPORTED 2 /* sizes outside the compiled tile shapes */
#define REPLAYSSM_ERR_MISALIGNED 3  /* a tensor pointer not 16-byte aligned */
#define REPLAYSSM_ERR_CUDA 4        /* the kernel launch reported an error */
#define REPLAYSSM_ERR_SCRATCH_LIMIT 5 /* sizes need more than the fixed no-alloc scratch */

/* Per-sequence device status bits, OR-ed into state->status[seq]. */
#define REPLAYSSM_SEQ_RING_FULL 1  /* decode/verify would overflow the ring */
#define REPLAYSSM_SEQ_BAD_ACCEPT 2 /* accept count m < 0, m > K or len + m > W */
#define REPLAYSSM_SEQ_TIMEOUT 4    /* a bounded wait expired; work skipped */
#define REPLAYSSM_SEQ_BAD_POINTER 8 /* head outside [0, W) or len outside [0, W]; untouched */

/* Layer kinds and element types. */
#define REPLAYSSM_MAMBA2 0
#define REPLAYSSM_GDN 1
#define REPLAYSSM_KDA 2
#define REPLAYSSM_F32 0
#define REPLAYSSM_BF16 1

/* Sizes of one SSM layer for a batch of sequences. */
typedef struct replayssm_dims {
  int32_t kind;     /* REPLAYSSM_MAMBA2, _GDN or _KDA */
  int32_t batch;    /* sequences */
  int32_t heads;    /* H */
  int32_t groups;   /* Mamba-2 B/C groups G (G divides H); 1 for delta kinds */
  int32_t dk;       /* columns of a state row: Mamba-2 N, delta d_k */
  int32_t dv;       /* rows of a head's state: Mamba-2 P, delta d_v */
  int32_t window;   /* W, ring entries per sequence */
  int32_t in_dtype; /* element type of the vector inputs and their ring copies */
} replayssm_dims;

/*
 * Device pointers of one layer's decode state (all caller-owned).
 * A Mamba-2 state uses ring_x, ring_B, ring_C, ring_dt; a delta state uses
 * ring_q, ring_k, ring_v, ring_alpha, ring_beta; the other ring pointers are
 * ignored. ring_C and ring_q are optional (NULL: not stored; the decode
 * arithmetic never reads them back). S_read NULL selects the FP32 read path.
 * At initialisation the caller zeroes ring_head, ring_len, status and sync
 * and fills S_ckpt (then calls replayssm_refresh_read_copy if S_read is set).
 * `sync` is scratch used by the kernels to order the per-sequence pointer
 * update after every block of that sequence has read it; each call leaves it
 * at zero. `work` is scratch for the per-head values a decode or verify call
 * derives from the ring before it streams the state (the buffer terms, the
 * decay, the swept query or the fold weights); it must hold
 * replayssm_workspace_bytes(dims, K) bytes for the largest K used with this
 * state, needs no initialisation and is overwritten by every decode and
 * verify call.
 */
typedef struct replayssm_state {
  float* S_ckpt;      /* f32 checkpoint, never rounded */
  void* S_read;       /* bf16 read copy or NULL */
  void* ring_x;       /* Mamba-2 [b, H, W, P]    in_dtype */
  void* ring_B;       /* Mamba-2 [b, W, G, N]    in_dtype */
  void* ring_C;       /* Mamba-2 [b, W, G, N]    in_dtype, optional */
  float* ring_dt;     /* Mamba-2 [b, H, Wd]      f32 */
  void* ring_q;       /* delta   [b, H, W, d_k]  in_dtype, optional */
  void* ring_k;       /* delta   [b, H, W, d_k]  in_dtype */
  void* ring_v;       /* delta   [b, H, W, d_v]  in_dtype */
  float* ring_alpha;  /* GDN [b, H, Wd]; KDA [b, H, W, d_k] f32 */
  float* ring_beta;   /* delta   [b, H, Wd]      f32 */
  int32_t* ring_head; /* slot of the oldest entry after the checkpoint */
  int32_t* ring_len;  /* committed entries after the checkpoint, 0..W */
  int32_t* status;    /* REPLAYSSM_SEQ_* bits; the library only sets bits */
  int32_t* sync;      /* scratch arrival counters, zero between calls */
  float* work;        /* scratch, replayssm_workspace_bytes(dims, K) bytes, any contents */
} replayssm_state;

/*
 * Mamba-2 replay decode of one token per sequence ("NVIDIA y Princeton
 * aceleran modelos híbridos…", paragraph 2: append, then output from the
 * checkpoint). Precondition per sequence: ring_len + 1 <= W (call
 * replayssm_consolidate(k_next = 1) first), else RING_FULL and the sequence
 * (ring, pointers, y) is untouched. Effects: writes the token into slot
 * (head + len) mod W, sets len += 1 and writes
 *   y = (prod_i dA_i) (h_c C) + sum_j w_j (C . B_j) x_j + D x,
 *   dA_i = exp(dt_i A), w_j = dt_j prod_{i > j} dA_i,
 * over the n = len + 1 buffered tokens, reading h_c from S_read (bf16) when
 * set, else S_ckpt. A, D: f32 [H]. No state is written.
 */
REPLAYSSM_API replayssm_status replayssm_mamba2_decode(
    const replayssm_dims* dims, const replayssm_state* state, const float* A, const float* D,
    const void* x, const void* B, const void* C, const float* dt, float* y, void* stream);

/*
 * Gated DeltaNet / KDA replay decode of one token per sequence (same page
 * and paragraph; layer kinds from "NVIDIA présente ReplaySSM…", section
 * "Pourquoi les hybrides sont devenus la norme"). dims->kind selects the
 * gate shape. Precondition and ring/pointer effects as for
 * replayssm_mamba2_decode. Output o = scale * S_t q, evaluated as
 *   u <- q; for j = n..1: s = k_j . u; o += beta_j s v_j;
 *           u <- alpha_j (elementwise) (u - beta_j s k_j);
 *   o += S_c u,
 * with A_j = Diag(alpha_j)(I - beta_j k_j k_j^T), S_t = S_{t-1} A_t + beta_t v_t k_t^T.
 */
REPLAYSSM_API replayssm_status replayssm_gdn_decode(
    const replayssm_dims* dims, const replayssm_state* state, const void* q, const void* k,
    const void* v, const float* alpha, const float* beta, float scale, float* o, void* stream);

/*
 * Consolidate ("NVIDIA y Princeton aceleran modelos híbridos…", paragraph 2:
 * the persistent state is only updated when the buffer fills; paragraph 4:
 * the recurrence runs at high precision, the read copy is refreshed from it).
 * For every sequence with len + k_next > W, or with force != 0 and len > 0,
 * folds its len committed entries into S_ckpt in FP32, writes S_ckpt once,
 * refreshes S_read = bf16_rne(S_ckpt) when S_read is set, and sets
 * head = (head + len) mod W, len = 0. Other sequences are untouched.
 * A: f32 [H] for Mamba-2, ignored (may be NULL) for the delta kinds.
 * k_next >= 0; force is 0 or 1.
 */
REPLAYSSM_API replayssm_status replayssm_consolidate(
    const replayssm_dims* dims, const replayssm_state* state, const float* A, int32_t k_next,
    int32_t force, void* stream);

/*
 * One plain decode step of a Mamba-2 layer with the consolidation it needs,
 * in one call: the result (outputs, S_ckpt, S_read, ring, pointers, status)
 * is that of replayssm_consolidate(dims, state, A, 1, 0) followed by
 * replayssm_mamba2_decode with the same arguments, up to float rounding
 * order. A sequence whose ring is full is folded as its state rows stream
 * past (the fold only when the buffer fills: "NVIDIA y Princeton aceleran
 * modelos híbridos…", paragraph 2): S_ckpt is read once and written once,
 * with S_read, and the output is computed from the new rows as the read
 * copy holds them. Every other sequence is decoded from S_read as by
 * replayssm_mamba2_decode. Arguments and layouts as for
 * replayssm_mamba2_decode; state->work must hold
 * replayssm_workspace_bytes(dims, 1) bytes and state->sync must be zero
 * (each call leaves it zero). With W > 16, or with a read copy whose row
 * block (about 16 KB of rows, at most P) is not a multiple of 64 rows -- P
 * of 32 or 96, say -- the call runs the fold and the decode as two launches
 * with the same result. Sequences with out-of-range pointers get
 * REPLAYSSM_SEQ_BAD_POINTER and are untouched. With the environment variable
 * REPLAYSSM_FOLD_TENSOR_CORES=1 the fold's rank-n update runs on the tensor
 * cores (mma.sync, TF32 operands split in hi + lo, three products per step,
 * about FP32 accuracy) instead of FP32 FMAs: a measured alternative, slower
 * on B300 at these shapes, kept for that comparison.
 */
REPLAYSSM_API replayssm_status replayssm_mamba2_fold_decode(
    const replayssm_dims* dims, const replayssm_state* state, const float* A, const float* D,
    const void* x, const void* B, const void* C, const float* dt, float* y, void* stream);

/*
 * One plain decode step of a Gated DeltaNet or KDA layer with the
 * consolidation it needs, in one call: the result (outputs, S_ckpt, S_read,
 * ring, pointers, status) is that of replayssm_consolidate(dims, state,
 * NULL, 1, 0) followed by replayssm_gdn_decode with the same arguments, up
 * to float rounding order. A sequence whose ring is full is folded and its
 * token decoded from the new rows ("NVIDIA y Princeton aceleran modelos
 * híbridos…", paragraph 2: the fold only when the buffer fills): S_ckpt is
 * read once and written once, with S_read, and the output comes from the
 * new rows as the read copy holds them, with no further read of the state.
 * Every other sequence is decoded as by replayssm_gdn_decode. Arguments and
 * layouts as for replayssm_gdn_decode; state->work must hold
 * replayssm_workspace_bytes(dims, 1) bytes (it carries one flag per
 * sequence between the two grids of the call) and state->sync must be zero
 * (each call leaves it zero). Sequences with out-of-range pointers get
 * REPLAYSSM_SEQ_BAD_POINTER and are untouched.
 */
REPLAYSSM_API replayssm_status replayssm_gdn_fold_decode(
    const replayssm_dims* dims, const replayssm_state* state, const void* q, const void* k,
    const void* v, const float* alpha, const float* beta, float scale, float* o, void* stream);

/*
 * Speculative verify for the delta kinds ("ReplaySSM: o ganho aparece…",
 * section "O que muda para quem desenvolve", and "NVIDIA y Princeton…",
 * paragraph 3: draft inputs are kept in the buffer, no state copy per
 * draft). Writes draft i (i < K) of each sequence into slot
 * (head + len + i) mod W without committing it, and outputs
 * o[:, i] = scale * S q_i for the state after the committed entries and
 * drafts 0..i, all K outputs from one read of the checkpoint. Draft fields
 * are [b, K, H, ...] (alpha [b, K, H] or [b, K, H, d_k], beta [b, K, H]).
 * Precondition len + K <= W (consolidate with k_next = K first), else
 * RING_FULL and the sequence is untouched. Mamba-2 layers use
 * replayssm_mamba2_spec_verify (here: REPLAYSSM_ERR_UNSUPPORTED).
 * GDN with a BF16 read copy and BF16 inputs (K > 1, W <= 16, d_k 64 or
 * 128, d_v a multiple of 64, state->S_read 16-byte aligned) runs the
 * tensor-core form: the products S [q_0..q_{K-1} | k_0..k_{n-1}]^T on
 * mma.sync (BF16 operands, FP32 sums) and the sweep coefficients from a
 * Gram tile of the keys; the environment variable
 * REPLAYSSM_DELTA_TENSOR_CORES=0 selects the FFMA kernel instead (same
 * results up to FP32 rounding order).
 */
REPLAYSSM_API replayssm_status replayssm_spec_verify(
    const replayssm_dims* dims, const replayssm_state* state, int32_t K, const void* q,
    const void* k, const void* v, const float* alpha, const float* beta, float scale, float* o,
    void* stream);

/*
 * Speculative verify for Mamba-2 layers (same passages as
 * replayssm_spec_verify; the pointer rollback applies to every SSM layer
 * type of "NVIDIA présente ReplaySSM…", "Pourquoi les hybrides sont devenus
 * la norme"). Writes draft i (i < K) of each sequence into slot
 * (head + len + i) mod W without committing it and outputs, for the state
 * after the committed entries and drafts 0..i, all from one read of the
 * checkpoint:
 *   y[:, i] = (prod dA) (h_c C_i) + sum_j w_j (C_i . B_j) x_j + D x_i.
 * Drafts: x [b, K, H, P], B and C [b, K, G, N] (in_dtype), dt [b, K, H] f32;
 * y [b, K, H, P] f32; A, D f32 [H]. state->work must hold
 * replayssm_workspace_bytes(dims, K) bytes. 1 <= K <= min(8, W).
 * Precondition len + K <= W (consolidate with k_next = K first), else
 * RING_FULL and the sequence is untouched. Accept with replayssm_accept.
 */
REPLAYSSM_API replayssm_status replayssm_mamba2_spec_verify(
    const replayssm_dims* dims, const replayssm_state* state, int32_t K, const float* A,
    const float* D, const void* x, const void* B, const void* C, const float* dt, float* y,
    void* stream);

/*
 * Accept the first m[s] verified drafts of each sequence by moving its
 * pointer: len += m[s] ("ReplaySSM: o ganho aparece…", section "O que muda
 * para quem desenvolve"; "NVIDIA y Princeton…", paragraph 3). m: int32 [b]
 * on the device. Requires 0 <= m <= K and len + m <= W, else BAD_ACCEPT and
 * no change. Rejected drafts stay in their slots until overwritten.
 */
REPLAYSSM_API replayssm_status replayssm_accept(
    const replayssm_dims* dims, const replayssm_state* state, const int32_t* m, int32_t K,
    void* stream);

/* S_read = bf16_rne(S_ckpt) for the whole batch (initialisation). S_read must be set. */
REPLAYSSM_API replayssm_status replayssm_refresh_read_copy(
    const replayssm_dims* dims, const replayssm_state* state, void* stream);

/*
 * Conventional per-token read-modify-write Mamba-2 step, the baseline the
 * method replaces ("ReplaySSM: o ganho aparece…", introduction: the whole
 * state matrix is read and written every token). S: f32 [b, H, P, N],
 * updated in place: h = exp(dt A) h + dt x B^T; y = h C + D x.
 */
REPLAYSSM_API replayssm_status replayssm_conventional_mamba2_step(
    const replayssm_dims* dims, float* S, const float* A, const float* D, const void* x,
    const void* B, const void* C, const float* dt, float* y, void* stream);

/*
 * Conventional per-token read-modify-write GDN/KDA step (same baseline).
 * S: f32 [b, H, d_v, d_k] updated in place: S = S A_t + beta v k^T;
 * o = scale * S q.
 */
REPLAYSSM_API replayssm_status replayssm_conventional_gdn_step(
    const replayssm_dims* dims, float* S, const void* q, const void* k, const void* v,
    const float* alpha, const float* beta, float scale, float* o, void* stream);

/*
 * Conventional speculative verify of K drafts with a state snapshot per
 * draft: the baseline that rollback by a buffer pointer replaces ("NVIDIA
 * présente ReplaySSM : accélérer le décodage des modèles hybrides Mamba et
 * GDN", section "D'où vient le problème de l'état": a fixed-size state cannot
 * be truncated, so each draft's state is kept). GDN/KDA only.
 * S: f32 [b, H, d_v, d_k], read, not modified. Drafts q, k, v [b, K, H, d]
 * (in_dtype), alpha [b, K, H] or [b, K, H, d_k], beta [b, K, H] (f32).
 * Writes snapshots[b, K, H, d_v, d_k] (f32), the state after drafts 0..i,
 * and o[b, K, H, d_v] = scale * S_i q_i. 1 <= K <= 8.
 */
REPLAYSSM_API replayssm_status replayssm_conventional_gdn_verify(
    const replayssm_dims* dims, const float* S, int32_t K, const void* q, const void* k,
    const void* v, const float* alpha, const float* beta, float scale, float* snapshots, float* o,
    void* stream);

/*
 * Conventional accept after replayssm_conventional_gdn_verify: for each
 * sequence, S = snapshot m[seq] - 1 (m = 0 leaves S unchanged). m outside
 * [0, K] sets REPLAYSSM_SEQ_BAD_ACCEPT in status[seq] (status may be NULL)
 * and leaves S unchanged. Any kind; S and snapshots as above (Mamba-2:
 * P x N per head). batch <= 65535.
 */
REPLAYSSM_API replayssm_status replayssm_conventional_accept(const replayssm_dims* dims, float* S,
                                                             const float* snapshots,
                                                             const int32_t* m, int32_t K,
                                                             int32_t* status, void* stream);

/*
 * Mamba-2 replay decode that allocates nothing and needs no caller scratch.
 * The pages have no counterpart: this is a library convenience.
 *
 * Some callers cannot allocate device memory when they decode: a plugin or
 * custom operator whose host framework owns all device memory and allows no
 * allocation inside its execution step, or a serving loop that reserved the
 * whole device for its state pool up front, where a late cudaMalloc can fail
 * and a cudaFree synchronizes the device. This entry point computes exactly
 * what replayssm_mamba2_decode computes, with the same arguments, but takes
 * its scratch -- the per-head workspace and the per-sequence arrival counters
 * that replayssm_mamba2_decode reads from state->work and state->sync -- from
 * one fixed array of REPLAYSSM_NOALLOC_SCRATCH_BYTES (16 MiB) in the
 * library's own device memory. state->work and state->sync are not read and
 * may be NULL; every other state field, input and output is as for
 * replayssm_mamba2_decode, and the caller still owns all of them.
 *
 * Limit: replayssm_mamba2_decode_noalloc_bytes(dims) bytes must not exceed
 * REPLAYSSM_NOALLOC_SCRATCH_BYTES, else the call returns
 * REPLAYSSM_ERR_SCRATCH_LIMIT before any CUDA call. That is the plain
 * decode's per-head rows, batch * heads * align4(P + 1) * 4 bytes, plus one
 * 4-byte flag per sequence rounded up to 16 bytes, rounded up to 256 bytes,
 * plus 4 * batch bytes of arrival counters. (Batch 256 x 128 heads at
 * P = 64 needs about 8.5 MiB.)
 *
 * The array exists once per GPU that loads the library and is held until the
 * process exits. Every call looks up the array's device address in the
 * current device's context (no call allocates). Each call clears the arrival
 * counters (the only part that must
 * start at zero) on `stream` before its kernels; the workspace rows and flags
 * are written before they are read. All calls share the one array, so calls
 * whose work overlaps on the GPU (other streams, other host threads) race and
 * give wrong results: serialize them, e.g. on one stream.
 */
REPLAYSSM_API replayssm_status replayssm_mamba2_decode_noalloc(
    const replayssm_dims* dims, const replayssm_state* state, const float* A, const float* D,
    const void* x, const void* B, const void* C, const float* dt, float* y, void* stream);

/* Size of the fixed scratch of replayssm_mamba2_decode_noalloc. */
#define REPLAYSSM_NOALLOC_SCRATCH_BYTES (16u << 20)

/*
 * Bytes of the fixed scratch that replayssm_mamba2_decode_noalloc needs for
 * these sizes (the formula above), so a caller can check the limit before
 * it calls; 0 if dims is invalid or not a Mamba-2 layer. Host only, no CUDA
 * call. The pages have no counterpart: a library convenience.
 */
REPLAYSSM_API int64_t replayssm_mamba2_decode_noalloc_bytes(const replayssm_dims* dims);

/*
 * Copies whole sequences between two layer states of the same dims: for each
 * i < n, sequence src_idx[i] of src is written to sequence dst_idx[i] of dst
 * (checkpoint, read copy, every ring field, ring head and len, status), so a
 * sequence resumes from (S_c, ring, pointer) without replaying its history
 * -- the state operations prefix caching and continuous batching need (the
 * pages' serving context, "NVIDIA présente ReplaySSM…", "D'où vient le
 * problème de l'état"). src and dst may be the same state (disjoint index
 * sets). Optional fields (S_read, ring_C / ring_q) must be set on both sides
 * or on neither. src_idx, dst_idx: device int32 [n], n <= 65535; pairs with
 * an index outside [0, batch) are skipped. Nothing may be in flight on
 * either state (the arrival counters are not copied and must be zero).
 */
REPLAYSSM_API replayssm_status replayssm_copy_sequences(const replayssm_dims* dims,
                                                       const replayssm_state* src,
                                                       const int32_t* src_idx,
                                                       const replayssm_state* dst,
                                                       const int32_t* dst_idx, int32_t n,
                                                       void* stream);

/*
 * Self-test of the kernels' bounded waits (no counterpart on the pages): one
 * warp waits on a barrier that nothing completes; after the wait limit (about
 * one second) it ORs REPLAYSSM_SEQ_TIMEOUT into status[0] and returns, and
 * the context stays usable. status: device int32, 16-byte aligned.
 */
REPLAYSSM_API replayssm_status replayssm_selftest_wait_timeout(int32_t* status, void* stream);

/*
 * Size in bytes of state->work for decode calls (K = 1; for Mamba-2 this
 * includes replayssm_mamba2_fold_decode's per-head weights) and verify
 * calls with up to K drafts on the given sizes (0 if dims is invalid).
 */
REPLAYSSM_API int64_t replayssm_workspace_bytes(const replayssm_dims* dims, int32_t K);

/*
 * Launch configuration of the persistent delta-rule kernel (GDN or KDA) that
 * replayssm_gdn_decode and the decode grid of replayssm_gdn_fold_decode
 * (K = 1) or replayssm_spec_verify (K drafts) would run for these sizes, on
 * a device whose blocks may use smem_limit bytes of shared memory (0: the
 * B300's 232,448). read_copy: 1 when the state has a BF16 read copy. Host
 * only, no CUDA call. It assumes the CUDA driver provides the tensor-map
 * encoder the tensor-core kernel needs; without it that kernel's calls run
 * the FFMA kernel instead. The pages have no counterpart: it reports how
 * the library lays one block out (prep warps staging heads, consumer groups
 * streaming state stages, the slots between them) so that the pipeline's
 * ownership rules can be checked without a GPU.
 * Returns REPLAYSSM_OK and fills *out; REPLAYSSM_ERR_INVALID_ARG for a NULL
 * pointer, invalid dims, a Mamba-2 layer, K outside [1, 8] or a negative
 * smem_limit; REPLAYSSM_ERR_UNSUPPORTED when no configuration fits.
 */
typedef struct replayssm_delta_config {
  int32_t tensor_cores;             /* 1: tensor-core verify kernel, 0: FFMA kernel */
  int32_t prep_warps;               /* NP */
  int32_t depth;                    /* heads staged per prep warp */
  int32_t state_stages;             /* NS, a multiple of consumer_groups */
  int32_t vector_slots;             /* FFMA kernel: NSL; tensor-core kernel: NP x depth */
  int32_t consumer_groups;          /* G */
  int32_t consumer_warps_per_group; /* GU */
  int32_t rows_per_unit;            /* state rows streamed per stage fill */
  int32_t units_per_head;           /* d_v / rows_per_unit */
  int32_t threads;                  /* per block */
  int64_t smem_bytes;               /* dynamic shared memory per block */
} replayssm_delta_config;

REPLAYSSM_API replayssm_status replayssm_delta_kernel_config(const replayssm_dims* dims,
                                                             int32_t K, int32_t read_copy,
                                                             int64_t smem_limit,
                                                             replayssm_delta_config* out);

/* Static, NUL-terminated description of a return code. */
REPLAYSSM_API const char* replayssm_status_string(replayssm_status status);

/* Library version as major * 10000 + minor * 100 + patch. */
REPLAYSSM_API int32_t replayssm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* REPLAYSSM_H */
