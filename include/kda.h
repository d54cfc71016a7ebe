/*
 * kda.h -- C ABI of the KDA recurrent-state hot path (libkda.so).
 *
 * What it computes.  Kimi Delta Attention keeps a fixed-size recurrent state
 * per (sequence, head) instead of a growing KV cache ("Confirmed" on the vLLM
 * Kimi K3 news page).  The pages name KDA but print no equation; this library
 * fixes it as a gated delta rule with per-key-channel decay:
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *     o_t = S_t^T q_t                                  (post-update state)
 *
 * S is d_k x d_v, alpha_t in R^{d_k} scales key rows, beta_t is a scalar.
 * No scaling of q and no normalisation of k happen inside the library.
 *
 * Three parts ("vLLM lifts Kimi K3 throughput by up to 2.8x"):
 *   - chunked prefill that exports state checkpoints at cache-block
 *     boundaries inside the same pass ("KDA checkpoints stay inside the
 *     prefill");
 *   - T-token draft verification over the committed state;
 *   - ReplaySSM commit: the drafted tokens' inputs are kept in a replay ring
 *     and the accepted state is rebuilt by replay, so a rejection only moves
 *     a pointer and no state is written per draft position ("ReplaySSM
 *     shrinks rollback state").
 * Mixed batches of speculative and ordinary requests use contiguous segments
 * of one packed token tensor and write outputs in place ("Small tensor copies
 * leave the hot path").
 *
 * Conventions for every entry point.
 *   - All pointers inside the structs and all int32 index arrays are DEVICE
 *     pointers unless stated; the caller owns every buffer.  The library
 *     allocates no device memory and keeps no per-call host state.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream).  Argument errors are detected on the host
 *     before anything is enqueued and returned synchronously as a negative
 *     status; nothing is launched then.
 *   - Errors that depend on device data (a slot id out of range, an accepted
 *     length above the pending count, a segment longer than the ring) are
 *     never trapped: the affected (sequence, head) unit is skipped, its state
 *     and ring are left untouched, and a KDA_DERR_* bit is ORed into a
 *     library-wide device error word read by kda_get_device_error().
 *   - Packed token tensors are [N][H][d] row-major (beta is [N][H]);
 *     sequence i owns rows [cu_seqlens[i], cu_seqlens[i+1]).
 *   - A state pool is fp32 [num_slots][H][d_v][d_k]: the state S of one
 *     (slot, head) is stored transposed, so each column of S (one value
 *     channel, all key channels) is contiguous.
 *   - Supported head dims: d_k == d_v in {16, 32, 64, 128}.  Input dtypes:
 *     fp32 or bf16 (q, k, v, alpha and beta all the same dtype); state and
 *     outputs are fp32.  Every pointer must be 16-byte aligned.
 *   - Calls that touch disjoint buffers may run concurrently on different
 *     streams; the device error word is shared.
 */
#ifndef KDA_H
#define KDA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *kda_stream_t;

/* Status codes (return values). */
enum {
  KDA_OK = 0,
  KDA_EINVAL = -1,  /* bad scalar argument or NULL pointer                */
  KDA_EDTYPE = -2,  /* unsupported or mismatched dtype                     */
  KDA_ESHAPE = -3,  /* unsupported or mismatched dimension                 */
  KDA_EALIGN = -4,  /* a pointer is not 16-byte aligned                    */
  KDA_EPROTO = -5,  /* ring / commit protocol misuse detectable on host    */
  KDA_ECUDA = -6,   /* a CUDA runtime call failed (launch, copy, sync)     */
  KDA_EDEVICE = -7, /* kda_get_device_error found bits set                 */
  KDA_ENOSPC = -8   /* workspace smaller than kda_prefill_workspace_size() */
};

/* Bits of the device error word. */
enum {
  KDA_DERR_SLOT = 1,     /* a state / checkpoint slot id outside the pool  */
  KDA_DERR_ACCEPT = 2,   /* accepted_len < 0 or above the pending count     */
  KDA_DERR_DEPTH = 4,    /* a speculative segment longer than ring depth    */
  KDA_DERR_SEGMENT = 8,  /* cu_seqlens not non-decreasing / beyond N        */
  KDA_DERR_RING = 16,    /* ring control word corrupt (pending > depth)     */
  KDA_DERR_RANGE = 32,   /* prefill: cumulative log-decay across half a
                            chunk below -80 in some channel (fp32 factor
                            range); outputs of that chunk are unreliable   */
  KDA_DERR_TIMEOUT = 64, /* a bounded wait (tensor cores, copy engine, a
                            pipeline stage) gave up; the kernel stopped
                            taking work: what it had not finished (outputs,
                            states, rings of those units) is left as it was
                            or unspecified, never half-written silently   */
  KDA_DERR_UNSAFE = 128  /* after a timeout, the second bounded wait for
                            work still in flight (tensor cores or copies)
                            also gave up before the kernel released its
                            tensor memory or shared memory; once
                            kda_get_device_error has seen this bit, every
                            later launching call on that device returns
                            KDA_EDEVICE for the rest of the process      */
};

typedef enum { KDA_F32 = 0, KDA_BF16 = 1 } kda_dtype;

/* One packed batch of tokens and its output buffer. */
typedef struct {
  kda_dtype dtype;          /* dtype of q, k, v, alpha, beta                */
  const void *q;            /* [N][H][d_k]                                  */
  const void *k;            /* [N][H][d_k]                                  */
  const void *v;            /* [N][H][d_v]                                  */
  const void *alpha;        /* [N][H][d_k]  per-channel decay in (0, 1]     */
  const void *beta;         /* [N][H]                                       */
  float *o;                 /* [N][H][d_v]  fp32 outputs, written in place  */
  const int32_t *cu_seqlens; /* [B + 1] device, cu[0] = 0, cu[B] = N        */
  int32_t num_seqs;         /* B                                            */
  int32_t num_tokens;       /* N (host copy of cu_seqlens[B])               */
  int32_t num_heads;        /* H                                            */
  int32_t d_k, d_v;
} kda_tokens;

/* Paged per-sequence states: fp32 [num_slots][H][d_v][d_k]. */
typedef struct {
  float *base;
  int32_t num_slots, num_heads, d_k, d_v;
} kda_state_pool;

/* ReplaySSM ring, one per state pool (per layer).  For every (slot, head)
 * it holds the inputs of the last verify's drafted tokens, entry e = the
 * e-th drafted position, plus a control pair {pending, accepted}:
 *   k, alpha : [num_slots][H][depth][d_k]   (token dtype)
 *   v        : [num_slots][H][depth][d_v]   (token dtype)
 *   beta     : [num_slots][H][depth]        (token dtype)
 *   ctrl     : [num_slots][H][2] int32      {pending, accepted}
 * A slot's ctrl must be zero (kda_ring_reset) before its first verify.
 * depth must be in [1, 16]. */
typedef struct {
  void *k, *v, *alpha, *beta;
  int32_t *ctrl;
  int32_t depth;
  kda_dtype dtype;
} kda_replay_ring;

/*
 * kda_prefill_chunked -- chunked prefill with in-pass checkpoints.
 * ("KDA checkpoints stay inside the prefill", vLLM Kimi K3 optimisation page.)
 *
 * For each sequence i the state starts at pool[state_slots[i]], runs every
 * token of segment i through the recurrence (chunk-wise WY/UT form, chunks
 * of `chunk` tokens aligned to absolute positions), writes o for every
 * token, and writes the final state back to pool[state_slots[i]].
 * Checkpoints: let p0 = start_pos[i] (tokens already folded into the state;
 * start_pos may be NULL = all zero).  After the token at absolute position
 * P = (floor(p0 / ckpt_every) + m + 1) * ckpt_every (1-based count of tokens
 * in the sequence) the state is copied into pool[ckpt_slots[i * max_ckpt + m]]
 * for m < max_ckpt; entries < 0 are skipped; boundaries past max_ckpt are
 * dropped.  ckpt_every == 0 disables checkpoints (ckpt_slots may be NULL).
 * Requirements: chunk in {16, 32, 64}; ckpt_every % chunk == 0; workspace of
 * at least kda_prefill_workspace_size(...) bytes, 256-byte aligned, owned by
 * the caller and not used by another call until this one completes.
 * At the tensor-core shape (bf16 inputs, d_k = d_v = 128, chunk 64, heads a
 * multiple of 8) the workspace is optional: with one, the chunks' state-
 * independent operands are computed for all chunks at once into it and a
 * second pass walks the chunks (the faster path for long sequences); with
 * NULL, one pass per (value slice, head, sequence) does everything.  Both
 * meet the same tolerances; they are not bit-identical to each other.
 * The target slots must have no pending commit (see kda_materialize).
 */
int kda_prefill_chunked(const kda_tokens *tok, kda_state_pool *pool,
                        const int32_t *state_slots, const int32_t *ckpt_slots,
                        int32_t max_ckpt, int32_t ckpt_every, int32_t chunk,
                        const int32_t *start_pos, void *workspace,
                        size_t workspace_bytes, kda_stream_t stream);

/*
 * kda_prefill_chunked_raw -- kda_prefill_chunked on projection-space inputs,
 * with the input-side preparation fused into the kernels instead of a
 * separate pass over the tokens (the pages leave the preparation open; it
 * follows the formulas the synthetic workloads are drawn with):
 *   k     : raw keys, L2-normalised over d_k per (token, head) in-kernel;
 *   alpha : decay logits z, alpha = exp(-softplus(z)) per key channel;
 *   beta  : logits b, beta = sigmoid(b) per (token, head);
 *   q, v  : used as given.
 * The prep runs in fp32 on the values as given (nothing is rounded to the
 * input dtype in between).  Only the tensor-core shape (bf16 inputs,
 * d_k = d_v = 128, chunk 64, heads a multiple of 8) is supported; other
 * shapes return KDA_ESHAPE.  Arguments and outputs otherwise as
 * kda_prefill_chunked (workspace optional at that shape).
 */
int kda_prefill_chunked_raw(const kda_tokens *tok, kda_state_pool *pool,
                            const int32_t *state_slots, const int32_t *ckpt_slots,
                            int32_t max_ckpt, int32_t ckpt_every, int32_t chunk,
                            const int32_t *start_pos, void *workspace,
                            size_t workspace_bytes, kda_stream_t stream);

/* Bytes of workspace kda_prefill_chunked needs for these sizes and input
 * dtype (at the tensor-core shape: for the two-pass path, about 162 KiB per
 * (chunk of 64 tokens, head)), and 0 on bad arguments (which the prefill call
 * itself rejects). */
size_t kda_prefill_workspace_size(int32_t num_tokens, int32_t num_seqs,
                                  int32_t num_heads, int32_t d_k, int32_t d_v,
                                  int32_t chunk, kda_dtype dtype);

/*
 * kda_prefill_chunked_noalloc -- kda_prefill_chunked for callers that cannot
 * allocate device memory.  (No counterpart on the pages: this is a service of
 * this library, not part of the method.)
 *
 * Some hosts own every byte of device memory through their own allocator and
 * forbid a library from calling cudaMalloc (or make it unsafe to do so while
 * their work is in flight), and some callers simply have no allocator handle
 * to pass a workspace from.  This entry point needs no workspace argument:
 * its scratch is a fixed array of KDA_NOALLOC_SCRATCH_BYTES in device memory
 * that belongs to this library, and every GPU that loads the library holds
 * that array until the process exits.  Nothing is allocated or freed here.
 *
 * Arguments, outputs and semantics are those of kda_prefill_chunked; the
 * caller still passes inputs, outputs, pool and slot tables.
 *   - Returns KDA_ENOSPC, before any CUDA call, when
 *     kda_prefill_workspace_size(...) for these sizes and dtype exceeds
 *     KDA_NOALLOC_SCRATCH_BYTES, except at the tensor-core shape, which then
 *     runs the single pass without touching the array.
 *   - The first call on a device looks up the array's device address (with
 *     that device current); make that first call before any stream capture.
 *     The address is kept for the life of the process: after a
 *     cudaDeviceReset it is stale (as is the device error word's), so do
 *     not call into the library again on a device that was reset.
 *   - Every call shares the one array and it keeps the last call's contents
 *     (no part of it needs to start at zero: each call writes what it reads).
 *     Calls whose work overlaps on the GPU (different streams, or different
 *     host threads, without ordering between them) race on it; order them.
 */
#define KDA_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
int kda_prefill_chunked_noalloc(const kda_tokens *tok, kda_state_pool *pool,
                                const int32_t *state_slots,
                                const int32_t *ckpt_slots, int32_t max_ckpt,
                                int32_t ckpt_every, int32_t chunk,
                                const int32_t *start_pos, kda_stream_t stream);

/*
 * kda_verify -- one verify launch over a mixed packed batch.
 * ("ReplaySSM shrinks rollback state"; "Small tensor copies leave the hot
 * path".)
 *
 * For every sequence i and head h, with slot s = state_slots[i]:
 *   1. the pending commit of (s, h) is applied first: the `accepted` leading
 *      ring entries recorded by the last kda_commit are replayed onto the
 *      state, token by token, and the state is written back once;
 *   2. speculative rows (is_spec[i] != 0, or is_spec == NULL): the segment's
 *      T_i <= max_T <= depth drafted tokens are evaluated from the committed
 *      state, o receives their outputs, their inputs are copied into ring
 *      entries 0..T_i-1, and ctrl becomes {T_i, 0}; no draft state is stored;
 *   3. ordinary rows (is_spec[i] == 0): the segment's tokens are applied and
 *      committed at once (ordinary decode), o receives their outputs, and
 *      ctrl becomes {0, 0}.
 * A verify that follows another verify with no kda_commit between them
 * treats the earlier drafts as all rejected.
 * The kernel is launched as a programmatic dependent of the previous work on
 * the stream: it may start while that work finishes, but it only prefetches
 * into L2 until that work has completed, so stream order holds for every
 * value it reads.  kda_materialize launches the same way.
 */
int kda_verify(const kda_tokens *tok, int32_t max_T, kda_state_pool *pool,
               const int32_t *state_slots, kda_replay_ring *ring,
               const int32_t *is_spec, kda_stream_t stream);

/*
 * kda_verify_raw -- kda_verify on projection-space inputs, the input prep
 * fused into the verify kernel (the fused-kernel direction of "Small tensor
 * copies leave the hot path"; the pages do not define the prep, so it
 * follows the formulas the synthetic workloads are drawn with, as
 * kda_prefill_chunked_raw does):
 *   k     : raw keys, L2-normalised over d_k per (token, head);
 *   alpha : decay logits z, alpha = exp(-softplus(z)) = 1 / (1 + e^z);
 *   beta  : logits b, beta = sigmoid(b);
 *   q, v  : used as given.
 * Precision: each token's prepared k, alpha and beta are computed once, in
 * IEEE fp32, when its row is loaded, and rounded to bf16 (round to nearest);
 * the drafts, ordinary decode and the ring entries all use those bf16 values,
 * so a replayed state equals the decoded one bit for bit and the ring holds
 * prepared inputs (a later kda_verify or kda_materialize replays it as usual).
 * Shapes: bf16 tokens, d_k = d_v = 128, ring depth <= 8, max_T <= 8; any
 * other shape returns KDA_ESHAPE before anything is launched.  Everything
 * else -- arguments, ownership, ordering, errors -- is kda_verify's.
 */
int kda_verify_raw(const kda_tokens *tok, int32_t max_T, kda_state_pool *pool,
                   const int32_t *state_slots, kda_replay_ring *ring,
                   const int32_t *is_spec, kda_stream_t stream);

/*
 * kda_forward_mixed -- one KDA layer over a packed batch that holds prefill
 * segments beside speculative and ordinary decode segments, read in place
 * with outputs written in place ("Small tensor copies leave the hot path":
 * contiguous zero-copy slices and direct output writes; "KDA checkpoints stay
 * inside the prefill").
 *
 * Sequences 0 .. num_prefill-1 of tok are prefill segments and occupy token
 * rows [0, prefill_tokens) (prefill_tokens = cu_seqlens[num_prefill], passed
 * on the host); they follow kda_prefill_chunked with state_slots[i],
 * ckpt_slots [num_prefill][max_ckpt], start_pos [num_prefill] (or NULL) and
 * the workspace (sized by kda_prefill_workspace_size(prefill_tokens,
 * num_prefill, ...); NULL allowed where kda_prefill_chunked allows it).
 * Sequences num_prefill .. num_seqs-1 follow kda_verify with
 * state_slots[num_prefill + j], is_spec[num_prefill + j] (is_spec indexed
 * over the whole batch, or NULL) and ring.  The parts must use distinct slots.
 * Results are those of the two separate calls, bit for bit.
 * With side_stream non-NULL (and not `stream`) the prefill part runs on
 * side_stream, forked from `stream` and joined back by events, beside the
 * verify part on `stream`; the call returns with `stream` ordered after both.
 * The two events are made once per host thread and device and reused by
 * every call (a stream capture of the call records their waits as graph
 * edges, as with any event).
 */
int kda_forward_mixed(const kda_tokens *tok, int32_t num_prefill, int32_t prefill_tokens,
                      kda_state_pool *pool, const int32_t *state_slots,
                      const int32_t *ckpt_slots, int32_t max_ckpt, int32_t ckpt_every,
                      int32_t chunk, const int32_t *start_pos, void *workspace,
                      size_t workspace_bytes, int32_t max_T, kda_replay_ring *ring,
                      const int32_t *is_spec, kda_stream_t stream,
                      kda_stream_t side_stream);

/*
 * kda_commit -- record how many drafted tokens each sequence accepted.
 * ("ReplaySSM shrinks rollback state", vLLM Kimi K3 optimisation page: a
 * rejection records a count and writes no state.)
 *
 * accepted_len[i] (device, 0 <= a <= pending) is recorded in ctrl of every
 * head of slot state_slots[i]; the replay itself is folded into the next
 * kda_verify or kda_materialize of that slot, so the state is read and
 * written once per step.  a == 0 leaves the state untouched.  No host sync.
 */
int kda_commit(const int32_t *accepted_len, const int32_t *state_slots,
               int32_t num_seqs, kda_state_pool *pool, kda_replay_ring *ring,
               kda_stream_t stream);

/*
 * kda_commit_layers -- kda_commit for the rings of several layers in one
 * launch: a speculative step verifies every KDA layer, samples once, and
 * records the same accepted_len[i] in each layer's ring.  rings is a HOST
 * array of num_layers <= 64 ring descriptors whose pools all have the
 * geometry of `pool` (the pool's base pointer is not used).
 */
int kda_commit_layers(const int32_t *accepted_len, const int32_t *state_slots,
                      int32_t num_seqs, const kda_state_pool *pool,
                      const kda_replay_ring *rings, int32_t num_layers,
                      kda_stream_t stream);

/*
 * kda_materialize -- apply every recorded commit now: replay the accepted
 * ring entries of each listed slot onto its state, write the state, and
 * clear ctrl to {0, 0}.  Call before reading a state any other way (gather,
 * copy, prefill from it) after a commit.  ("ReplaySSM shrinks rollback
 * state": the accepted state is rebuilt from the kept inputs; this is that
 * rebuild on demand, for a state about to be read outside a verify.)
 */
int kda_materialize(const int32_t *state_slots, int32_t num_seqs,
                    kda_state_pool *pool, kda_replay_ring *ring,
                    kda_stream_t stream);

/* kda_ring_reset -- set ctrl of every head of the listed slots to {0, 0}
 * (a fresh slot, or drafts to discard: "ReplaySSM shrinks rollback state",
 * where discarding drafts is a pointer move, not a state write). */
int kda_ring_reset(const int32_t *slots, int32_t n, const kda_state_pool *pool,
                   kda_replay_ring *ring, kda_stream_t stream);

/* kda_gather_states -- out[i] = pool[slots[i]] for i < n; out is fp32
 * [n][H][d_v][d_k] on the device.  Reads committed-and-materialized state.
 * (Paged per-sequence state addressed through a slot table: the hybrid
 * cache of the daily.dev Kimi K3 summary, and "KDA checkpoints stay inside
 * the prefill", whose checkpoints are read back by slot.) */
int kda_gather_states(const kda_state_pool *pool, const int32_t *slots,
                      int32_t n, float *out, kda_stream_t stream);

/* kda_copy_slots -- pool[dst[i]] = pool[src[i]] for i < n (prefix-cache
 * fork of a checkpoint into a live slot: "KDA checkpoints stay inside the
 * prefill", where a partial prefix hit resumes from a block-boundary
 * checkpoint).  The src and dst sets must be disjoint. */
int kda_copy_slots(kda_state_pool *pool, const int32_t *src,
                   const int32_t *dst, int32_t n, kda_stream_t stream);

/*
 * kda_verify_snapshot -- the direct design that ReplaySSM replaces, kept as
 * an ablation baseline ("ReplaySSM shrinks rollback state": storing the
 * state at every drafted position costs T state writes per step).
 *
 * For every sequence i and head h, with slot s = state_slots[i] and the
 * segment's T_i <= max_T <= 16 drafted tokens: the state of (s, h) is
 * advanced token by token, o receives each token's output, and the state
 * after drafted token t (0-based) is written to snapshot (i, t):
 *   snapshots: device fp32 [num_seqs][max_T][H][d_v][d_k] (each snapshot in
 *   the pool's per-slot layout), owned by the caller; entries t >= T_i are
 *   not written.
 * The pool is only read.  Snapshot (i, t) holds the same bits as the state
 * that a ReplaySSM commit of t + 1 tokens rebuilds from the same state and
 * inputs.  The slots must have no pending ReplaySSM commit.  A segment
 * longer than max_T sets KDA_DERR_DEPTH and skips the sequence.
 */
int kda_verify_snapshot(const kda_tokens *tok, int32_t max_T,
                        const kda_state_pool *pool, const int32_t *state_slots,
                        float *snapshots, kda_stream_t stream);

/*
 * kda_commit_snapshot -- commit of the direct design: for every sequence i
 * with a = accepted_len[i] > 0 (device), every head of pool[state_slots[i]]
 * receives snapshot (i, a - 1) of the preceding kda_verify_snapshot (same
 * max_T); a == 0 leaves the state untouched.  a must not exceed that
 * verify's T_i; a < 0 or a > max_T sets KDA_DERR_ACCEPT and skips the row.
 */
int kda_commit_snapshot(const int32_t *accepted_len, const int32_t *state_slots,
                        int32_t num_seqs, kda_state_pool *pool,
                        const float *snapshots, int32_t max_T,
                        kda_stream_t stream);

/* kda_get_device_error -- synchronize `stream`, read the device error word
 * of the current device into *host_bits (host pointer), clear it, and return
 * KDA_EDEVICE if any bit was set, else KDA_OK. */
int kda_get_device_error(int32_t *host_bits, kda_stream_t stream);

/* kda_set_wait_limit -- testing hook for the failure path: every bounded
 * device wait of later launches (tensor-core completions, pipeline stages,
 * copy arrivals) gives up after `polls` polls instead of the default
 * (about 4 M polls), and reports KDA_DERR_TIMEOUT; a negative value restores
 * the default.  With polls = 0 a kernel's first wait gives up at once: the
 * pipelined verify then writes nothing (no output, state, ring or ctrl
 * word) and still lets its own copies land before it exits.  The second,
 * drain-before-exit waits keep their own fixed limit.  Library-wide, not
 * per stream; meant for tests, not for serving. */
int kda_set_wait_limit(int32_t polls);

/* Human-readable name of a status code (static string). */
const char *kda_status_string(int status);

/* Library ABI version: 1. */
int kda_version(void);

#ifdef __cplusplus
}
#endif
#endif /* KDA_H */
