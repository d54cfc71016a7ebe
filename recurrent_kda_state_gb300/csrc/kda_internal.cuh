// Internal declarations shared by the CUDA translation units of libkda.so.
// Launch parameter blocks, device-side dtype helpers and the launchers that
// kda_api.cu calls after validating the public arguments.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

// ----------------------------------------------------------------- dtypes
template <typename Tin>
struct InVec;  // 16-byte vector of inputs, converted to fp32

template <>
struct InVec<float> {
  static constexpr int kElems = 4;
  __device__ __forceinline__ static void load(const float *p, float *dst) {
    const float4 a = *reinterpret_cast<const float4 *>(p);
    dst[0] = a.x; dst[1] = a.y; dst[2] = a.z; dst[3] = a.w;
  }
};

template <>
struct InVec<__nv_bfloat16> {
  static constexpr int kElems = 8;
  __device__ __forceinline__ static void load(const __nv_bfloat16 *p, float *dst) {
    const uint4 a = *reinterpret_cast<const uint4 *>(p);
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      dst[2 * i] = __uint_as_float(w[i] << 16);
      dst[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
};

template <typename Tin>
__device__ __forceinline__ float in_scalar(const Tin *p);
template <>
__device__ __forceinline__ float in_scalar<float>(const float *p) { return *p; }
template <>
__device__ __forceinline__ float in_scalar<__nv_bfloat16>(const __nv_bfloat16 *p) {
  return __bfloat162float(*p);
}
__device__ __forceinline__ void set_error(unsigned int *err, unsigned int bit) {
  atomicOr(err, bit);
}

// ------------------------------------------------------- launch parameters
struct VerifyParams {
  const void *q, *k, *v, *alpha, *beta;  // packed inputs (NULL when mode==1)
  float *o;
  const int32_t *cu_seqlens;
  const int32_t *state_slots;
  const int32_t *is_spec;  // may be NULL (all speculative)
  float *pool;
  void *rk, *rv, *ra, *rb;  // ring payload
  int32_t *ctrl;            // ring control [P][H][2]
  unsigned int *err;
  int B, N, H, P, depth, max_T;
  int mode;             // 0 = verify, 1 = materialize (no tokens)
  int prefetch_stride;  // CTAs of the first wave (0: no L2 prefetch)
  int spin_limit;       // polls of a bounded wait before it gives up
  int raw;              // tokens are projections: prep applied in-kernel
};

struct CommitParams {
  const int32_t *accepted_len;  // NULL for ring reset
  const int32_t *slots;
  int32_t *ctrl;
  unsigned int *err;
  int B, H, P;
};

constexpr int kMaxCommitLayers = 64;
struct CommitLayersParams {
  const int32_t *accepted_len;
  const int32_t *slots;
  int32_t *ctrl[kMaxCommitLayers];
  unsigned int *err;
  int B, H, P, L;
};

// Direct per-position snapshots (the design ReplaySSM replaces): verify that
// stores the state after every drafted token, and a commit that copies the
// accepted one into the pool.
struct SnapshotParams {
  const void *q, *k, *v, *alpha, *beta;
  float *o;
  const int32_t *cu_seqlens;
  const int32_t *state_slots;
  const int32_t *accepted_len;  // commit only
  float *pool;
  float *snap;                  // [B][max_T][H][d_v][d_k]
  unsigned int *err;
  int B, N, H, P, max_T;
};

struct SlotCopyParams {
  const float *src_base;
  float *dst_base;
  const int32_t *src_slots;  // indices into src_base's pool
  const int32_t *dst_slots;  // NULL: dst is dense [n][state]
  unsigned int *err;
  int n, P;
  long long state_floats;  // H * d_v * d_k
};

struct PrefillParams {
  const void *q, *k, *v, *alpha, *beta;
  float *o;
  const int32_t *cu_seqlens;
  const int32_t *state_slots;
  const int32_t *ckpt_slots;  // [B][max_ckpt] or NULL
  const int32_t *start_pos;   // [B] or NULL
  float *pool;
  unsigned char *ws;          // workspace (chunk table + per-chunk operands)
  unsigned int *err;
  int B, N, H, P, max_ckpt, ckpt_every, max_chunks;
  int raw;  // inputs are projections: k unnormalised, alpha and beta logits
  int spin_limit;  // polls of a bounded wait before it gives up
};

// Workspace geometry of the chunked prefill (shared with the size query):
// [chunk table: (B + 1) int32, padded to 256 B][entries: (chunk, head) ->
// prefill_entry_floats(D, C) fp32 each, 256-byte aligned].
__host__ __device__ inline size_t prefill_table_bytes(int B) {
  return ((size_t)(B + 1) * sizeof(int) + 255) & ~(size_t)255;
}
__host__ __device__ inline size_t prefill_entry_floats(int D, int C) {
  const size_t f = (size_t)4 * C * D + (size_t)C * C + D;
  return (f + 63) & ~(size_t)63;
}
__host__ __device__ inline int prefill_max_chunks(int N, int B, int C) {
  return N / C + 2 * B;
}
// The tensor-core prefill (no workspace) takes bf16 inputs at d_k = d_v = 128,
// chunk 64, with a head count that is a multiple of 8; other shapes run the
// CUDA-core kernels on the caller's workspace.
__host__ __device__ inline bool prefill_uses_tc(int dtype, int H, int d_k, int d_v,
                                                int C) {
  return dtype == KDA_BF16 && d_k == 128 && d_v == 128 && C == 64 && H % 8 == 0;
}
__host__ __device__ inline size_t prefill_workspace_bytes(int N, int B, int H,
                                                          int D, int C) {
  return prefill_table_bytes(B) + (size_t)prefill_max_chunks(N, B, C) * H *
                                      prefill_entry_floats(D, C) * sizeof(float);
}
// Two-pass tensor-core prefill (the tensor-core shape with a workspace): the
// chunk table, then per (chunk, head) one entry of kTcEntryBytes holding the
// chunk's state-independent operands as shared-memory images (see
// kda_prefill_tc.cu), entries 1024-byte aligned from the workspace base.
constexpr size_t kTcEntryBytes = 165888;
__host__ __device__ inline size_t prefill_tc_entries_offset(int B) {
  return (prefill_table_bytes(B) + 1023) & ~(size_t)1023;
}
__host__ __device__ inline size_t prefill_tc_workspace_bytes(int N, int B, int H) {
  return prefill_tc_entries_offset(B) +
         (size_t)prefill_max_chunks(N, B, 64) * H * kTcEntryBytes;
}

// Chunk g of the workspace chunk table (prefix sums of the sequences' chunk
// counts): its sequence, its index in the sequence, and its rows.
struct ChunkLoc {
  int i, q, tok0, n, end_local, L, p0;
};
__device__ __forceinline__ ChunkLoc locate_chunk(const PrefillParams &p, int g,
                                                 int C) {
  const int *table = reinterpret_cast<const int *>(p.ws);
  int lo = 0, hi = p.B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (table[mid] <= g) lo = mid; else hi = mid - 1;
  }
  ChunkLoc c;
  c.i = lo;
  c.q = g - table[lo];
  c.L = p.cu_seqlens[lo + 1] - p.cu_seqlens[lo];
  c.p0 = p.start_pos ? p.start_pos[lo] : 0;
  const int r = c.p0 % C;
  const int s_loc = max(0, c.q * C - r);
  c.end_local = min(c.L, (c.q + 1) * C - r);
  c.n = c.end_local - s_loc;
  c.tok0 = p.cu_seqlens[lo] + s_loc;
  return c;
}

// Polls of a bounded wait on the tensor cores or the copy engine before it
// gives up (KDA_DERR_TIMEOUT): the library's default, or the value a test set
// through kda_set_wait_limit.  The second, drain-before-exit wait of a kernel
// always uses kDrainWaitPolls.
constexpr int kDefaultWaitPolls = 1 << 22;
constexpr int kDrainWaitPolls = 1 << 26;
int wait_limit_polls();

// The argument checks of kda_prefill_chunked that do not concern the
// workspace (pool, tokens, chunk, checkpoints, slot table); KDA_OK or the
// status that call would return.
int prefill_check_args(const kda_tokens *tok, kda_state_pool *pool,
                       const int32_t *state_slots, const int32_t *ckpt_slots,
                       int32_t max_ckpt, int32_t ckpt_every, int32_t chunk);

// Verify launch geometry: dynamic shared memory for (D, ring depth, max_T),
// and the longest speculative segment the kernel supports (ring depth limit).
size_t verify_smem_bytes(int D, int depth, int max_T, kda_dtype dt);
int verify_max_spec_tokens();

// Launchers: return cudaError_t of the launch.
cudaError_t launch_verify(const VerifyParams &p, kda_dtype dt, int D,
                          cudaStream_t s);
// The pipelined verify kernel (d = 128, bf16, ring depth <= 8, <= 8 tokens
// per row): whether it serves these parameters, and its launcher.
bool verify_pipe_applies(const VerifyParams &p, kda_dtype dt, int D);
cudaError_t launch_verify_pipe(const VerifyParams &p, cudaStream_t s);
cudaError_t launch_commit(const CommitParams &p, cudaStream_t s);
cudaError_t launch_commit_layers(const CommitLayersParams &p, cudaStream_t s);
cudaError_t launch_ring_reset(const CommitParams &p, cudaStream_t s);
cudaError_t launch_slot_copy(const SlotCopyParams &p, cudaStream_t s);
cudaError_t launch_verify_snapshot(const SnapshotParams &p, kda_dtype dt, int D,
                                   cudaStream_t s);
cudaError_t launch_commit_snapshot(const SnapshotParams &p, int D, cudaStream_t s);
cudaError_t launch_prefill(const PrefillParams &p, kda_dtype dt, int D, int C,
                           cudaStream_t s);
// Tensor-core prefill (d_k = d_v = 128, chunk 64, bf16 inputs, heads a
// multiple of 8): two passes through the workspace when p.ws is set, else one
// pass with no workspace.
cudaError_t launch_prefill_tc(const PrefillParams &p, cudaStream_t s);
// The chunk table at the start of the workspace (one thread).
cudaError_t launch_chunk_table(const PrefillParams &p, int C, cudaStream_t s);

}  // namespace kda
