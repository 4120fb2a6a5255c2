/*
 * gdn.h -- C ABI of the GB300 (sm_103a) chunked Gated Delta Rule prefill library.
 *
 * The one operation: the varlen, packed Gated Delta Rule prefill scan.  For each
 * sequence n (token rows [cu_seqlens[n], cu_seqlens[n+1])) and each sab head h,
 * starting from the state S (128 x 128, V-major: row = value index, column = key
 * index), every token t updates and reads the state:
 *
 *     S_t = g_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *     o_t = scale S_t q_t
 *
 * Sources: the operation and its arguments are those of
 * flashinfer.cudnn.cudnn_chunk_gated_delta_rule (Parameters; Returns) and of
 * flashinfer.chunk_gated_delta_rule ("flashinfer.gdn_prefill": the chunked GDN
 * scan that initialises the recurrent state from a full prompt before decode).
 * The state layout and the state-dtype pass-through are from "flashinfer.cudnn",
 * Linear attention.  The split-K partition and batch invariance are from the
 * batch_invariant parameter of cudnn_chunk_gated_delta_rule.
 *
 * Conventions for every entry point:
 *  - Tensors are described by gdn_tensor_t: a data pointer, a dtype, a rank and
 *    per-dimension sizes and strides counted in ELEMENTS.  Data pointers are
 *    DEVICE pointers on the current device.
 *  - The caller owns every buffer.  The library never frees or keeps a pointer
 *    past the call.  All work is enqueued on `stream`; nothing is synchronised,
 *    so results are valid once the stream has reached the call.
 *  - Errors: every entry point returns a gdn_status_t.  On any error detected on
 *    the host nothing is launched and nothing is written.  gdn_last_error()
 *    returns a message describing the most recent error of the calling thread.
 *  - Inputs the host cannot see (the contents of cu_seqlens and state_indices)
 *    are checked on the device: a sequence with a negative, decreasing or
 *    out-of-range bound, or a state index outside the pool, is skipped (its
 *    output rows and state slot are not written) and a device error word is
 *    set; read it with gdn_get_device_status().  No kernel traps.
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARGUMENT = 1, /* null required tensor, wrong rank/shape/stride, bad scale */
    GDN_ERR_UNSUPPORTED = 2,      /* dtype, head_dim != 128, head-count relation or device arch */
    GDN_ERR_ALIAS = 3,            /* an output overlaps an input it must not alias */
    GDN_ERR_CUDA = 4,             /* a CUDA runtime / driver call failed */
    GDN_ERR_DEVICE_INPUT = 5      /* device-detected bad cu_seqlens / state index / timeout */
} gdn_status_t;

typedef enum {
    GDN_F32 = 0,
    GDN_BF16 = 1,
    GDN_F16 = 2,
    GDN_I32 = 3,
    GDN_I64 = 4
} gdn_dtype_t;

/* A strided tensor view.  `stride` is in elements; unused trailing dims are ignored. */
typedef struct {
    void* data;
    int32_t dtype;      /* gdn_dtype_t */
    int32_t ndim;
    int64_t shape[4];
    int64_t stride[4];
} gdn_tensor_t;

/* Bits of the device error word returned by gdn_get_device_status(). */
#define GDN_DEVERR_CU_SEQLENS   0x1  /* some cu_seqlens bound was negative, decreasing or > T */
#define GDN_DEVERR_STATE_INDEX  0x2  /* some state_indices entry was outside the state pool */
#define GDN_DEVERR_TIMEOUT      0x4  /* an on-chip wait gave up (the unit's results are invalid) */

/*
 * gdn_init: check that `device` is an sm_103 GPU (compute capability 10.3) and
 * set up per-device state.  Called lazily by gdn_chunk_prefill for the current
 * device; calling it explicitly moves the check to start-up, as the availability
 * check at backend initialisation of "[perf]FlashInfer cuDNN batched prefill
 * attention" (Availability checks) does, so that an unusable installation fails when
 * the backend is set up rather than on the first call.  Returns GDN_ERR_UNSUPPORTED on
 * any other architecture: unsupported architectures fail closed, with no fallback
 * ("flashinfer.gdn_prefill", Cake GDN CP context-parallel backend).
 */
gdn_status_t gdn_init(int device);

/*
 * gdn_chunk_prefill: chunked Gated Delta Rule prefill over a packed varlen batch.
 * Argument order and meaning follow cudnn_chunk_gated_delta_rule (Parameters).
 *
 *  q, k           [T, H_qk, 128] bf16 or f16 (q, k, v one dtype; with f16 every
 *                 tensor-core operand is f16).  Innermost dim contiguous; the token and
 *                 head strides are free (e.g. slices of a fused qkv buffer) but
 *                 must be positive multiples of 8 elements, and the base 16-byte
 *                 aligned (they are read through TMA).  q and k have equal shapes.
 *  v              [T, H_v, 128], q's dtype, same stride rules.
 *                 H = max(H_qk, H_v) sab heads; H must be a multiple of both.
 *                 Sab head h reads q/k head h / (H / H_qk) and v head h / (H / H_v).
 *  g              nullable.  [T, H] forget gate in LINEAR space (alpha = exp(log g)),
 *                 f32, bf16 or f16, any strides.  NULL means all ones.
 *                 Values are expected in (0, 1]; g below the smallest positive
 *                 normal float is treated as that float, and g above 1 as 1.
 *  beta           nullable.  [T, H] post-sigmoid update gate, f32, bf16 or f16, any
 *                 strides.  NULL means all ones.
 *  scale          query scale; 0 means 1/sqrt(128).  Must be finite.
 *  initial_state  nullable.  [slots, H, 128, 128] f32, bf16 or f16, V-major; the inner
 *                 128 x 128 block contiguous, slot/head strides free.  NULL means
 *                 every sequence starts from the zero state.
 *  state_indices  nullable.  [N] i32 or i64: sequence n reads initial_state slot
 *                 state_indices[n] and writes output_state slot state_indices[n].
 *                 NULL means slot n.  Slots must be unique (caller precondition).
 *  output_state   nullable.  [slots, H, 128, 128] f32, bf16 or f16 (same layout rules
 *                 as initial_state); receives the final state of each sequence,
 *                 rounded to its own dtype.  NULL writes no state at all.  It must
 *                 not overlap initial_state (GDN_ERR_ALIAS): split-K CTAs read the
 *                 incoming state while others write the outgoing one.
 *  cu_seqlens     [N + 1] i32 or i64, contiguous, required.  Sequence n covers
 *                 token rows [cu_seqlens[n], cu_seqlens[n+1]); empty sequences are
 *                 allowed (their final state is their initial state).
 *  use_qk_l2norm  nonzero: q and k rows are divided by sqrt(sum(x^2) + 1e-6) first.
 *  batch_invariant nonzero: never split a sequence across CTAs, so every output
 *                 and state bit depends only on that sequence's own inputs.
 *                 Zero: the library may split every sequence into P segments of
 *                 whole 64-token chunks (P = 1..8, equal segments or a skewed plan,
 *                 picked from the number of (sequence, head) units, the mean length
 *                 and the SM count; P = 1 whenever splitting would not pay;
 *                 gdn_testing_split_plan shows the plan).  With P > 1 the call enqueues
 *                 three kernels: pass 1 runs segment 0 and, for every middle
 *                 segment p, its affine state map S -> S M_p + N_p; a fix-up
 *                 chains S_{p+1} = S_p M_p + N_p in f32; pass 2 runs segments
 *                 1..P-1 from those states.  Results are deterministic for a given
 *                 batch but not bit-identical across batchings.  The maps live in a
 *                 library-owned workspace of N * H * (3P - 5) * 64 KiB per device,
 *                 grown with cudaMallocAsync on `stream` (the old one released with
 *                 cudaFreeAsync) and freed by gdn_shutdown(); split calls on two
 *                 streams of one device must not run concurrently.  While `stream`
 *                 is being captured into a CUDA graph the workspace is not grown:
 *                 the call fails with GDN_ERR_UNSUPPORTED unless
 *                 gdn_reserve_workspace made it large enough beforehand.
 *                 gdn_testing_force_splits forces P, for tests.
 *  output         [T, H, 128] in q's dtype, innermost contiguous, written in place.  Must
 *                 not overlap q, k, v or the states (GDN_ERR_ALIAS).
 *  stream         the CUDA stream all work is enqueued on.
 */
gdn_status_t gdn_chunk_prefill(const gdn_tensor_t* q, const gdn_tensor_t* k,
                               const gdn_tensor_t* v, const gdn_tensor_t* g,
                               const gdn_tensor_t* beta, float scale,
                               const gdn_tensor_t* initial_state,
                               const gdn_tensor_t* state_indices,
                               const gdn_tensor_t* output_state,
                               const gdn_tensor_t* cu_seqlens, int use_qk_l2norm,
                               int batch_invariant, const gdn_tensor_t* output,
                               cudaStream_t stream);

/*
 * gdn_chunk_prefill_checkpointed: gdn_chunk_prefill that also writes mid-sequence f32
 * state checkpoints (the "checkpoints" of the Cake GDN CP input domain in
 * "flashinfer.gdn_prefill", FP32 checkpoints; for prefix caching).  Same arguments,
 * validation and results as gdn_chunk_prefill, plus:
 *  checkpoints         [N * M, H, 128, 128] f32, V-major, inner block contiguous, rows
 *                      16-byte aligned; block n * M + m, head h receives the state of
 *                      sequence n after its first (m + 1) * checkpoint_every * 64 tokens,
 *                      when the sequence is at least that long; other blocks are left
 *                      untouched.  Must not overlap any other argument (GDN_ERR_ALIAS).
 *  checkpoints_per_seq M >= 1.
 *  checkpoint_every    the checkpoint stride in 64-token chunks, >= 1.
 */
gdn_status_t gdn_chunk_prefill_checkpointed(const gdn_tensor_t* q, const gdn_tensor_t* k,
                                            const gdn_tensor_t* v, const gdn_tensor_t* g,
                                            const gdn_tensor_t* beta, float scale,
                                            const gdn_tensor_t* initial_state,
                                            const gdn_tensor_t* state_indices,
                                            const gdn_tensor_t* output_state,
                                            const gdn_tensor_t* cu_seqlens, int use_qk_l2norm,
                                            int batch_invariant, const gdn_tensor_t* output,
                                            const gdn_tensor_t* checkpoints, int checkpoints_per_seq,
                                            int checkpoint_every, cudaStream_t stream);

/*
 * gdn_decode_step: one token per batch row through the same recurrence, updating each
 * row's state slot in place -- the decode loop that the prefill's final state seeds
 * ("flashinfer.gdn_prefill": the chunked scan initialises the recurrent state from a
 * full prompt before decode takes over).  For row b and sab head h, with S the slot's
 * state (V-major) and k, q optionally L2-normalised:
 *
 *     S <- g S (I - beta k k^T) + beta v k^T,     o = scale S q
 *
 *  q, k           [B, H_qk, 128], v [B, H_v, 128], bf16 or f16 (same rules as
 *                 gdn_chunk_prefill's q/k/v, with B rows in place of T tokens).
 *  g, beta        nullable, [B, H]; as in gdn_chunk_prefill (g clamped to
 *                 [FLT_MIN, 1]; NULL means ones).
 *  scale          0 means 1/sqrt(128).
 *  state          [slots, H, 128, 128] f32, bf16 or f16 (inner block contiguous, rows 16-byte
 *                 aligned), read and written IN PLACE; required.
 *  state_indices  nullable [B] i32/i64: row b uses slot state_indices[b] (NULL: slot b).
 *                 Slots must be unique (caller precondition: duplicates race).  An
 *                 out-of-range index sets GDN_DEVERR_STATE_INDEX and skips the row.
 *  use_qk_l2norm  as in gdn_chunk_prefill.
 *  output         [B, H, 128] in q's dtype, innermost contiguous.
 * Errors as for gdn_chunk_prefill (the state must not overlap the other inputs or the
 * output: GDN_ERR_ALIAS).  Asynchronous on `stream`; no workspace.
 */
gdn_status_t gdn_decode_step(const gdn_tensor_t* q, const gdn_tensor_t* k, const gdn_tensor_t* v,
                             const gdn_tensor_t* g, const gdn_tensor_t* beta, float scale,
                             const gdn_tensor_t* state, const gdn_tensor_t* state_indices,
                             int use_qk_l2norm, const gdn_tensor_t* output, cudaStream_t stream);

/*
 * gdn_chunk_prefill_noalloc: the same operation, arguments, validation and
 * results as gdn_chunk_prefill, for callers that must not have the library
 * allocate device memory (the pages define no counterpart: it is an interface of
 * this library only).
 *
 *  - Scratch: a fixed static device array of the library module, 256 B of header
 *    plus 32 MiB of split-K workspace (512 blocks of 128 x 128 f32).  The call
 *    makes no cudaMalloc/cudaFree or other allocating call.  A batch_invariant = 0
 *    call whose split needs more than 32 MiB (N * H * (3P - 5) * 64 KiB) fails
 *    with GDN_ERR_UNSUPPORTED before anything is enqueued; batch_invariant = 1
 *    never needs workspace.
 *  - Set-up: the first call on a device checks the device and looks up the
 *    scratch address (cudaGetSymbolAddress, with that device current); later
 *    calls reuse it.  Make that first call before any stream capture.
 *  - device_error: nullable DEVICE pointer to a caller-owned int32 into which the
 *    kernels OR the GDN_DEVERR_* bits (never cleared by the library).  NULL: the
 *    bits go to a word of the scratch header that is cleared on `stream` at the
 *    start of the call and is not reported.  gdn_get_device_status does not see
 *    this entry point's errors.
 *  - Concurrency: every call on a device shares the one scratch, so two calls
 *    that overlap in time (different streams, or different host threads) race on
 *    it.  Serialise them, e.g. on one stream.
 */
gdn_status_t gdn_chunk_prefill_noalloc(const gdn_tensor_t* q, const gdn_tensor_t* k,
                                       const gdn_tensor_t* v, const gdn_tensor_t* g,
                                       const gdn_tensor_t* beta, float scale,
                                       const gdn_tensor_t* initial_state,
                                       const gdn_tensor_t* state_indices,
                                       const gdn_tensor_t* output_state,
                                       const gdn_tensor_t* cu_seqlens, int use_qk_l2norm,
                                       int batch_invariant, const gdn_tensor_t* output,
                                       int32_t* device_error, cudaStream_t stream);

/*
 * Library memory management (the pages define no such call; the split-K workspace it
 * manages is the state-fixup scratch of cudnn_chunk_gated_delta_rule's split-K path,
 * "flashinfer.cudnn.cudnn_chunk_gated_delta_rule", Parameters, batch_invariant).
 *
 * gdn_reserve_workspace: grow the current device's split-K workspace to at least
 * `bytes` now, with cudaMallocAsync on `stream` (the previous block released with
 * cudaFreeAsync on the same stream), so that later gdn_chunk_prefill calls with
 * batch_invariant = 0 allocate nothing -- for instance while a CUDA graph is being
 * captured, when the library refuses to grow it (GDN_ERR_UNSUPPORTED).  The workspace
 * is owned by the library, never shrinks, and is freed by gdn_shutdown.  Returns
 * GDN_ERR_CUDA (message in gdn_last_error) if the allocation fails; the old workspace
 * is then gone too, and the next split call allocates again.
 *
 * gdn_split_workspace_bytes: the workspace bytes of a call with `splits` segments per
 * sequence, N * H * (3 * splits - 5) * 64 KiB; 0 for splits < 2 or non-positive sizes.
 * The planner never picks more than 8 segments, so gdn_split_workspace_bytes(N, H, 8)
 * covers every split of N sequences and H sab heads.  Pure host arithmetic.
 */
gdn_status_t gdn_reserve_workspace(size_t bytes, cudaStream_t stream);
size_t gdn_split_workspace_bytes(int64_t num_seqs, int64_t num_sab_heads, int splits);

/*
 * gdn_get_device_status: synchronise `stream`, then return in *device_error the
 * bits (GDN_DEVERR_*) that kernels on the current device have set since the last
 * call, and clear them.  Returns GDN_ERR_DEVICE_INPUT when any bit was set.  This is
 * how inputs the host never sees (cu_seqlens, state_indices) fail closed without a
 * trap ("flashinfer.gdn_prefill", Cake GDN CP context-parallel backend: invalid inputs
 * fail closed).
 */
gdn_status_t gdn_get_device_status(cudaStream_t stream, int32_t* device_error);

/*
 * Thread-local message of the calling thread's most recent error ("" if none): the
 * reason a call was declined, the counterpart of the per-engine reason that lands in
 * the frontend's log when an engine declines a graph
 * ("flashinfer.cudnn.cudnn_chunk_gated_delta_rule"; "flashinfer.cudnn", Linear
 * attention).
 */
const char* gdn_last_error(void);

/*
 * Release per-device library state: the device error words, the split-K workspace,
 * the cached address of the allocation-free entry's static scratch (looked up again on
 * that entry's next call; it is valid only as long as the CUDA context) and every
 * thread's cached launch settings (kernel attributes and SM counts, set up again on the
 * next launch), so that the library works again after a cudaDeviceReset that follows
 * the shutdown.  Safe to call more than once; call it with no work of the library in
 * flight.
 */
void gdn_shutdown(void);

/*
 * Testing aids (the pages define no such calls).  Both settings belong to the calling
 * host thread and apply to its later prefill calls; they are not meant for production.
 *
 * gdn_testing_force_splits: with `splits` in 1..8, calls with batch_invariant = 0 use
 * that many segments per sequence instead of the planner's choice, so that every
 * split-K layout can be exercised; 0 restores the planner.  GDN_ERR_INVALID_ARGUMENT
 * outside 0..8.
 *
 * gdn_testing_wait_limit: bound every on-chip hand-off wait of the prefill kernel by
 * `limit_ns` nanoseconds instead of the default 200 ms (0 restores the default; values
 * from 1 to 999 are refused with GDN_ERR_INVALID_ARGUMENT).  With
 * `withhold_local_ready` nonzero, the chunk-local group of every CTA withholds its
 * first "operands ready" hand-off, so that the wait for it runs out: the call then
 * returns normally, its results are invalid, and the device error word gets
 * GDN_DEVERR_TIMEOUT.  The waits that drain in-flight copies and MMAs before the CTA
 * exits keep the full bound either way.
 *
 * gdn_testing_split_plan: the split-K plan that gdn_chunk_prefill would take with
 * batch_invariant = 0 for `num_seqs` sequences of `total_tokens` tokens in all,
 * `num_heads` sab heads and `num_sms` SMs (the forced segment count of this thread
 * applies).  Host only, no GPU needed.  `plan` (int32[16], caller-owned) receives
 * P at [0], the segment denominator at [1], the segment numerators num[0..P] at [2..],
 * the grid of pass 1 and pass 2 at [11] and [12], and their unit counts at [13] and
 * [14]; segment p holds chunks [C num[p] / den, C num[p + 1] / den) of a C-chunk
 * sequence.  When P > 1, `units` (int32[2][capacity][2], caller-owned) receives for
 * every unit index u of pass 1 (block 0) and pass 2 (block 1) its (sequence * num_heads
 * + head, kind) pair, or (-1, -1) for an index that holds no unit; CTA u mod grid walks
 * index u.  Kinds of pass 1: 0 = segment 0, p in 1..P-2 = map M_p, P - 2 + p = map N_p;
 * of pass 2: kind k = segment k + 1.  GDN_ERR_INVALID_ARGUMENT for non-positive sizes,
 * or when `capacity` is below a pass's unit count.
 */
gdn_status_t gdn_testing_force_splits(int splits);
gdn_status_t gdn_testing_wait_limit(uint64_t limit_ns, int withhold_local_ready);
gdn_status_t gdn_testing_split_plan(int64_t num_seqs, int64_t num_heads, int64_t total_tokens,
                                    int num_sms, int32_t* plan, int32_t* units, int64_t capacity);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
