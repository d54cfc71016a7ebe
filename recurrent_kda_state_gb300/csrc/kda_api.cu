// Public C ABI of libkda.so: argument validation on the host, then launches on
// the caller's stream.  Nothing is allocated here; every buffer belongs to the
// caller.  The only library-owned device object is one error word per device.
#include <atomic>
#include <mutex>

#include "kda_internal.cuh"

// Library-wide device error word (one per device that loads the library).
__device__ unsigned int g_kda_device_error = 0;

namespace {

// Device address of g_kda_device_error for the current device.
unsigned int *device_error_word() {
  static std::mutex mu;
  static unsigned int *cache[64] = {};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_kda_device_error) != cudaSuccess) return nullptr;
    cache[dev] = static_cast<unsigned int *>(p);
  }
  return cache[dev];
}

// Polls of a bounded device wait (kda_set_wait_limit; negative = default).
std::atomic<int> g_wait_limit{-1};

// Devices on which a kernel reported KDA_DERR_UNSAFE (seen by
// kda_get_device_error): the library refuses further launches there.
std::atomic<unsigned long long> g_unsafe_devices{0};

bool device_unsafe() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  return (g_unsafe_devices.load() >> dev) & 1ull;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// The fork and join events of kda_forward_mixed on the current device, made
// once per host thread and device and reused by every call (a wait enqueued
// on an event takes the event's state at that moment, so re-recording it for
// the next call is safe).  nullptr if they could not be made.
cudaEvent_t *fork_events() {
  thread_local cudaEvent_t ev[64][2] = {};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (!ev[dev][0]) {
    if (cudaEventCreateWithFlags(&ev[dev][0], cudaEventDisableTiming) != cudaSuccess)
      return nullptr;
    if (cudaEventCreateWithFlags(&ev[dev][1], cudaEventDisableTiming) != cudaSuccess) {
      cudaEventDestroy(ev[dev][0]);
      ev[dev][0] = nullptr;
      return nullptr;
    }
  }
  return ev[dev];
}
bool dim_ok(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }
int cuda_status(cudaError_t e) { return e == cudaSuccess ? KDA_OK : KDA_ECUDA; }

constexpr int kMaxGridY = 65535;
constexpr size_t kMaxSmem = 227 * 1024;

int check_pool(const kda_state_pool *pool) {
  if (!pool || !pool->base) return KDA_EINVAL;
  if (!aligned16(pool->base)) return KDA_EALIGN;
  if (pool->num_slots < 1 || pool->num_heads < 1) return KDA_ESHAPE;
  if (pool->d_k != pool->d_v || !dim_ok(pool->d_k)) return KDA_ESHAPE;
  return KDA_OK;
}

int check_tokens(const kda_tokens *t, const kda_state_pool *pool, bool cu_aligned = true) {
  if (!t) return KDA_EINVAL;
  if (t->dtype != KDA_F32 && t->dtype != KDA_BF16) return KDA_EDTYPE;
  if (t->num_seqs < 0 || t->num_tokens < 0) return KDA_EINVAL;
  if (t->num_heads != pool->num_heads || t->d_k != pool->d_k || t->d_v != pool->d_v)
    return KDA_ESHAPE;
  if (t->num_seqs > kMaxGridY) return KDA_ESHAPE;
  if (t->num_seqs == 0) return KDA_OK;
  if (!t->cu_seqlens) return KDA_EINVAL;
  if (t->num_tokens > 0) {
    const void *ptrs[] = {t->q, t->k, t->v, t->alpha, t->beta, t->o};
    for (const void *p : ptrs) {
      if (!p) return KDA_EINVAL;
      if (!aligned16(p)) return KDA_EALIGN;
    }
  }
  if (cu_aligned && !aligned16(t->cu_seqlens)) return KDA_EALIGN;
  return KDA_OK;
}

int check_ring(const kda_replay_ring *r, kda_dtype dt, bool payload) {
  if (!r || !r->ctrl) return KDA_EINVAL;
  if (!aligned16(r->ctrl)) return KDA_EALIGN;
  if (r->depth < 1 || r->depth > kda::verify_max_spec_tokens()) return KDA_EINVAL;
  if (!payload) return KDA_OK;
  if (r->dtype != dt) return KDA_EDTYPE;
  const void *ptrs[] = {r->k, r->v, r->alpha, r->beta};
  for (const void *p : ptrs) {
    if (!p) return KDA_EINVAL;
    if (!aligned16(p)) return KDA_EALIGN;
  }
  return KDA_OK;
}

kda::VerifyParams verify_params(const kda_state_pool *pool,
                                const kda_replay_ring *ring,
                                const int32_t *slots, int B, unsigned *err) {
  kda::VerifyParams p = {};
  p.state_slots = slots;
  p.pool = pool->base;
  p.rk = ring->k;
  p.rv = ring->v;
  p.ra = ring->alpha;
  p.rb = ring->beta;
  p.ctrl = ring->ctrl;
  p.err = err;
  p.B = B;
  p.H = pool->num_heads;
  p.P = pool->num_slots;
  p.depth = ring->depth;
  p.spin_limit = kda::wait_limit_polls();
  return p;
}

}  // namespace

namespace kda {
int wait_limit_polls() {
  const int v = g_wait_limit.load();
  return v < 0 ? kDefaultWaitPolls : v;
}
}  // namespace kda

extern "C" {

int kda_version(void) { return 1; }

int kda_set_wait_limit(int32_t polls) {
  g_wait_limit.store(polls < 0 ? -1 : polls);
  return KDA_OK;
}

const char *kda_status_string(int status) {
  switch (status) {
    case KDA_OK: return "KDA_OK";
    case KDA_EINVAL: return "KDA_EINVAL: bad scalar argument or NULL pointer";
    case KDA_EDTYPE: return "KDA_EDTYPE: unsupported or mismatched dtype";
    case KDA_ESHAPE: return "KDA_ESHAPE: unsupported or mismatched dimension";
    case KDA_EALIGN: return "KDA_EALIGN: pointer not 16-byte aligned";
    case KDA_EPROTO: return "KDA_EPROTO: ring/commit protocol misuse";
    case KDA_ECUDA: return "KDA_ECUDA: CUDA runtime error";
    case KDA_EDEVICE: return "KDA_EDEVICE: device error bits set";
    case KDA_ENOSPC: return "KDA_ENOSPC: workspace too small";
    default: return "KDA_UNKNOWN";
  }
}

size_t kda_prefill_workspace_size(int32_t num_tokens, int32_t num_seqs,
                                  int32_t num_heads, int32_t d_k, int32_t d_v,
                                  int32_t chunk, kda_dtype dtype) {
  if (num_tokens < 0 || num_seqs < 0 || num_heads < 1 || d_k != d_v ||
      !dim_ok(d_k) || (chunk != 16 && chunk != 32 && chunk != 64) ||
      (dtype != KDA_F32 && dtype != KDA_BF16))
    return 0;
  if (kda::prefill_uses_tc(dtype, num_heads, d_k, d_v, chunk))
    return kda::prefill_tc_workspace_bytes(num_tokens, num_seqs, num_heads);
  return kda::prefill_workspace_bytes(num_tokens, num_seqs, num_heads, d_k, chunk);
}

}  // extern "C"

namespace {

int prefill_impl(const kda_tokens *tok, kda_state_pool *pool, const int32_t *state_slots,
                 const int32_t *ckpt_slots, int32_t max_ckpt, int32_t ckpt_every,
                 int32_t chunk, const int32_t *start_pos, void *workspace,
                 size_t workspace_bytes, kda_stream_t stream, bool cu_aligned,
                 bool raw = false, bool check_only = false) {
  int st = check_pool(pool);
  if (st) return st;
  if ((st = check_tokens(tok, pool, cu_aligned))) return st;
  if (chunk != 16 && chunk != 32 && chunk != 64) return KDA_EINVAL;
  if (ckpt_every < 0 || max_ckpt < 0) return KDA_EINVAL;
  if (ckpt_every > 0 && ckpt_every % chunk != 0) return KDA_EINVAL;
  if (ckpt_every > 0 && max_ckpt > 0 && !ckpt_slots) return KDA_EINVAL;
  if (tok->num_seqs == 0) return KDA_OK;
  if (!state_slots) return KDA_EINVAL;
  const bool tc = kda::prefill_uses_tc(tok->dtype, tok->num_heads, tok->d_k, tok->d_v, chunk);
  if (raw && !tc) return KDA_ESHAPE;  // the prep is fused into the tensor-core kernels
  if (check_only) return KDA_OK;
  // the CUDA-core kernels and the two-pass tensor-core kernels work in the
  // caller's workspace; at the tensor-core shape a NULL workspace selects the
  // single pass
  if (!tc && !workspace) return KDA_EINVAL;
  if (workspace) {
    if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return KDA_EALIGN;
    const size_t need =
        tc ? kda::prefill_tc_workspace_bytes(tok->num_tokens, tok->num_seqs, tok->num_heads)
           : kda::prefill_workspace_bytes(tok->num_tokens, tok->num_seqs, tok->num_heads,
                                          tok->d_k, chunk);
    if (workspace_bytes < need) return KDA_ENOSPC;
  }
  if ((long long)tok->num_tokens / chunk + 2LL * tok->num_seqs > 0x7fffffffLL)
    return KDA_ESHAPE;
  if (device_unsafe()) return KDA_EDEVICE;
  unsigned *err = device_error_word();
  if (!err) return KDA_ECUDA;
  kda::PrefillParams p = {};
  p.q = tok->q;
  p.k = tok->k;
  p.v = tok->v;
  p.alpha = tok->alpha;
  p.beta = tok->beta;
  p.o = tok->o;
  p.cu_seqlens = tok->cu_seqlens;
  p.state_slots = state_slots;
  p.ckpt_slots = ckpt_every > 0 && max_ckpt > 0 ? ckpt_slots : nullptr;
  p.start_pos = start_pos;
  p.pool = pool->base;
  p.ws = static_cast<unsigned char *>(workspace);
  p.err = err;
  p.B = tok->num_seqs;
  p.N = tok->num_tokens;
  p.H = tok->num_heads;
  p.P = pool->num_slots;
  p.max_ckpt = max_ckpt;
  p.ckpt_every = ckpt_every;
  p.max_chunks = kda::prefill_max_chunks(tok->num_tokens, tok->num_seqs, chunk);
  p.raw = raw ? 1 : 0;
  p.spin_limit = kda::wait_limit_polls();
  return cuda_status(kda::launch_prefill(p, tok->dtype, tok->d_k, chunk,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

int verify_impl(const kda_tokens *tok, int32_t max_T, kda_state_pool *pool,
                const int32_t *state_slots, kda_replay_ring *ring, const int32_t *is_spec,
                kda_stream_t stream, bool cu_aligned, bool raw = false) {
  int st = check_pool(pool);
  if (st) return st;
  if ((st = check_tokens(tok, pool, cu_aligned))) return st;
  if ((st = check_ring(ring, tok->dtype, true))) return st;
  if (max_T < 0) return KDA_EINVAL;
  if (!is_spec && max_T > ring->depth) return KDA_EPROTO;
  // the prep is fused into the pipelined kernel only
  if (raw && !(tok->dtype == KDA_BF16 && tok->d_k == 128 && tok->d_v == 128 &&
               ring->depth <= 8 && max_T <= 8))
    return KDA_ESHAPE;
  if (kda::verify_smem_bytes(tok->d_k, ring->depth, max_T, tok->dtype) > kMaxSmem)
    return KDA_EINVAL;
  if (tok->num_seqs == 0) return KDA_OK;
  if (!state_slots) return KDA_EINVAL;
  if (device_unsafe()) return KDA_EDEVICE;
  unsigned *err = device_error_word();
  if (!err) return KDA_ECUDA;
  kda::VerifyParams p = verify_params(pool, ring, state_slots, tok->num_seqs, err);
  p.q = tok->q;
  p.k = tok->k;
  p.v = tok->v;
  p.alpha = tok->alpha;
  p.beta = tok->beta;
  p.o = tok->o;
  p.cu_seqlens = tok->cu_seqlens;
  p.is_spec = is_spec;
  p.N = tok->num_tokens;
  p.max_T = max_T;
  p.mode = 0;
  p.raw = raw ? 1 : 0;
  return cuda_status(kda::launch_verify(p, tok->dtype, tok->d_k,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

}  // namespace

namespace kda {
int prefill_check_args(const kda_tokens *tok, kda_state_pool *pool,
                       const int32_t *state_slots, const int32_t *ckpt_slots,
                       int32_t max_ckpt, int32_t ckpt_every, int32_t chunk) {
  return prefill_impl(tok, pool, state_slots, ckpt_slots, max_ckpt, ckpt_every, chunk,
                      nullptr, nullptr, 0, nullptr, true, false, true);
}
}  // namespace kda

extern "C" {

int kda_prefill_chunked(const kda_tokens *tok, kda_state_pool *pool,
                        const int32_t *state_slots, const int32_t *ckpt_slots,
                        int32_t max_ckpt, int32_t ckpt_every, int32_t chunk,
                        const int32_t *start_pos, void *workspace,
                        size_t workspace_bytes, kda_stream_t stream) {
  return prefill_impl(tok, pool, state_slots, ckpt_slots, max_ckpt, ckpt_every, chunk,
                      start_pos, workspace, workspace_bytes, stream, true);
}

int kda_prefill_chunked_raw(const kda_tokens *tok, kda_state_pool *pool,
                            const int32_t *state_slots, const int32_t *ckpt_slots,
                            int32_t max_ckpt, int32_t ckpt_every, int32_t chunk,
                            const int32_t *start_pos, void *workspace,
                            size_t workspace_bytes, kda_stream_t stream) {
  return prefill_impl(tok, pool, state_slots, ckpt_slots, max_ckpt, ckpt_every, chunk,
                      start_pos, workspace, workspace_bytes, stream, true, true);
}

int kda_verify(const kda_tokens *tok, int32_t max_T, kda_state_pool *pool,
               const int32_t *state_slots, kda_replay_ring *ring,
               const int32_t *is_spec, kda_stream_t stream) {
  return verify_impl(tok, max_T, pool, state_slots, ring, is_spec, stream, true);
}

int kda_verify_raw(const kda_tokens *tok, int32_t max_T, kda_state_pool *pool,
                   const int32_t *state_slots, kda_replay_ring *ring,
                   const int32_t *is_spec, kda_stream_t stream) {
  return verify_impl(tok, max_T, pool, state_slots, ring, is_spec, stream, true, true);
}

int kda_forward_mixed(const kda_tokens *tok, int32_t num_prefill, int32_t prefill_tokens,
                      kda_state_pool *pool, const int32_t *state_slots,
                      const int32_t *ckpt_slots, int32_t max_ckpt, int32_t ckpt_every,
                      int32_t chunk, const int32_t *start_pos, void *workspace,
                      size_t workspace_bytes, int32_t max_T, kda_replay_ring *ring,
                      const int32_t *is_spec, kda_stream_t stream,
                      kda_stream_t side_stream) {
  int st = check_pool(pool);
  if (st) return st;
  if ((st = check_tokens(tok, pool))) return st;
  if (num_prefill < 0 || num_prefill > tok->num_seqs) return KDA_EINVAL;
  if (prefill_tokens < 0 || prefill_tokens > tok->num_tokens) return KDA_EINVAL;
  if (num_prefill == 0 && prefill_tokens != 0) return KDA_EINVAL;
  if (tok->num_seqs > 0 && !state_slots) return KDA_EINVAL;
  // the two parts: zero-copy views of the same packed tensors
  kda_tokens tp = *tok, tv = *tok;
  tp.num_seqs = num_prefill;
  tp.num_tokens = prefill_tokens;
  tv.num_seqs = tok->num_seqs - num_prefill;
  tv.cu_seqlens = tok->cu_seqlens ? tok->cu_seqlens + num_prefill : nullptr;
  if (tv.num_seqs > 0) {  // validate the verify part before anything is launched
    if ((st = check_ring(ring, tok->dtype, true))) return st;
    if (max_T < 0) return KDA_EINVAL;
    if (!is_spec && max_T > ring->depth) return KDA_EPROTO;
    if (kda::verify_smem_bytes(tok->d_k, ring->depth, max_T, tok->dtype) > kMaxSmem)
      return KDA_EINVAL;
  }
  const bool fork = side_stream != nullptr && side_stream != stream && num_prefill > 0 &&
                    tv.num_seqs > 0;
  cudaStream_t main_s = reinterpret_cast<cudaStream_t>(stream);
  cudaStream_t side_s = reinterpret_cast<cudaStream_t>(side_stream);
  cudaEvent_t *ev = nullptr;
  if (fork) {
    ev = fork_events();
    if (!ev || cudaEventRecord(ev[0], main_s) != cudaSuccess ||
        cudaStreamWaitEvent(side_s, ev[0], 0) != cudaSuccess)
      return KDA_ECUDA;
  }
  bool join = false;
  if (num_prefill > 0) {
    st = prefill_impl(&tp, pool, state_slots, ckpt_slots, max_ckpt, ckpt_every, chunk,
                      start_pos, workspace, workspace_bytes, fork ? side_stream : stream,
                      true);
    if (fork) {
      if (cudaEventRecord(ev[1], side_s) == cudaSuccess) join = true;
      else if (st == KDA_OK) st = KDA_ECUDA;
    }
  }
  if (st == KDA_OK && tv.num_seqs > 0)
    st = verify_impl(&tv, max_T, pool, state_slots + num_prefill, ring,
                     is_spec ? is_spec + num_prefill : nullptr, stream, false);
  if (fork) {
    // the caller's stream waits for whatever the side stream took (the join)
    if (join && cudaStreamWaitEvent(main_s, ev[1], 0) != cudaSuccess && st == KDA_OK)
      st = KDA_ECUDA;
  }
  return st;
}

int kda_commit(const int32_t *accepted_len, const int32_t *state_slots,
               int32_t num_seqs, kda_state_pool *pool, kda_replay_ring *ring,
               kda_stream_t stream) {
  int st = check_pool(pool);
  if (st) return st;
  if ((st = check_ring(ring, KDA_F32, false))) return st;
  if (num_seqs < 0) return KDA_EINVAL;
  if (num_seqs == 0) return KDA_OK;
  if (!accepted_len || !state_slots) return KDA_EINVAL;
  if (device_unsafe()) return KDA_EDEVICE;
  unsigned *err = device_error_word();
  if (!err) return KDA_ECUDA;
  kda::CommitParams p = {accepted_len, state_slots, ring->ctrl, err, num_seqs,
                         pool->num_heads, pool->num_slots};
  return cuda_status(kda::launch_commit(p, reinterpret_cast<cudaStream_t>(stream)));
}

int kda_commit_layers(const int32_t *accepted_len, const int32_t *state_slots,
                      int32_t num_seqs, const kda_state_pool *pool,
                      const kda_replay_ring *rings, int32_t num_layers,
                      kda_stream_t stream) {
  int st = check_pool(pool);
  if (st) return st;
  if (num_seqs < 0 || num_layers < 0 || num_layers > kda::kMaxCommitLayers)
    return KDA_EINVAL;
  if (num_seqs == 0 || num_layers == 0) return KDA_OK;
  if (!accepted_len || !state_slots || !rings) return KDA_EINVAL;
  kda::CommitLayersParams p = {};
  for (int l = 0; l < num_layers; ++l) {
    if ((st = check_ring(&rings[l], KDA_F32, false))) return st;
    p.ctrl[l] = rings[l].ctrl;
  }
  if (device_unsafe()) return KDA_EDEVICE;
  unsigned *err = device_error_word();
  if (!err) return KDA_ECUDA;
  p.accepted_len = accepted_len;
  p.slots = state_slots;
  p.err = err;
  p.B = num_seqs;
  p.H = pool->num_heads;
  p.P = pool->num_slots;
  p.L = num_layers;
  return cuda_status(
      kda::launch_commit_layers(p, reinterpret_cast<cudaStream_t>(stream)));
}

int kda_materialize(const int32_t *state_slots, int32_t num_seqs,
                    kda_state_pool *pool, kda_replay_ring *ring,
                    kda_stream_t stream) {
  int st = check_pool(pool);
  if (st) return st;
  if (!ring) return KDA_EINVAL;
  if ((st = check_ring(ring, ring->dtype, true))) return st;
  if (ring->dtype != KDA_F32 && ring->dtype != KDA_BF16) return KDA_EDTYPE;
  if (num_seqs < 0 || num_seqs > kMaxGridY) return KDA_EINVAL;
  if (num_seqs == 0) return KDA_OK;
  if (!state_slots) return KDA_EINVAL;
  if (device_unsafe()) return KDA_EDEVICE;
  unsigned *err = device_error_word();
  if (!err) return KDA_ECUDA;
  kda::VerifyParams p = verify_params(pool, ring, state_slots, num_seqs, err);
  p.max_T = 0;
  p.mode = 1;
  return cuda_status(kda::launch_verify(p, ring->dtype, pool->d_k,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

int kda_ring_reset(const int32_t *slots, int32_t n, const kda_state_pool *pool,
                   kda_replay_ring *ring, kda_stream_t stream) {
  int st = check_pool(pool);
  if (st) return st;
  if ((st = check_ring(ring, KDA_F32, false))) return st;
  if (n < 0) return KDA_EINVAL;
  if (n == 0) return KDA_OK;
  if (!slots) return KDA_EINVAL;
  if (device_unsafe()) return KDA_EDEVICE;
  unsigned *err = device_error_word();
  if (!err) return KDA_ECUDA;
  kda::CommitParams p = {nullptr, slots, ring->ctrl, err, n, pool->num_heads,
                         pool->num_slots};
  return cuda_status(kda::launch_ring_reset(p, reinterpret_cast<cudaStream_t>(stream)));
}

int kda_gather_states(const kda_state_pool *pool, const int32_t *slots,
                      int32_t n, float *out, kda_stream_t stream) {
  int st = check_pool(pool);
  if (st) return st;
  if (n < 0 || n > kMaxGridY) return KDA_EINVAL;
  if (n == 0) return KDA_OK;
  if (!slots || !out) return KDA_EINVAL;
  if (!aligned16(out)) return KDA_EALIGN;
  if (device_unsafe()) return KDA_EDEVICE;
  unsigned *err = device_error_word();
  if (!err) return KDA_ECUDA;
  kda::SlotCopyParams p = {};
  p.src_base = pool->base;
  p.dst_base = out;
  p.src_slots = slots;
  p.dst_slots = nullptr;
  p.err = err;
  p.n = n;
  p.P = pool->num_slots;
  p.state_floats = (long long)pool->num_heads * pool->d_v * pool->d_k;
  return cuda_status(kda::launch_slot_copy(p, reinterpret_cast<cudaStream_t>(stream)));
}

int kda_copy_slots(kda_state_pool *pool, const int32_t *src, const int32_t *dst,
                   int32_t n, kda_stream_t stream) {
  int st = check_pool(pool);
  if (st) return st;
  if (n < 0 || n > kMaxGridY) return KDA_EINVAL;
  if (n == 0) return KDA_OK;
  if (!src || !dst) return KDA_EINVAL;
  if (device_unsafe()) return KDA_EDEVICE;
  unsigned *err = device_error_word();
  if (!err) return KDA_ECUDA;
  kda::SlotCopyParams p = {};
  p.src_base = pool->base;
  p.dst_base = pool->base;
  p.src_slots = src;
  p.dst_slots = dst;
  p.err = err;
  p.n = n;
  p.P = pool->num_slots;
  p.state_floats = (long long)pool->num_heads * pool->d_v * pool->d_k;
  return cuda_status(kda::launch_slot_copy(p, reinterpret_cast<cudaStream_t>(stream)));
}

int kda_verify_snapshot(const kda_tokens *tok, int32_t max_T,
                        const kda_state_pool *pool, const int32_t *state_slots,
                        float *snapshots, kda_stream_t stream) {
  int st = check_pool(pool);
  if (st) return st;
  if ((st = check_tokens(tok, pool))) return st;
  if (max_T < 1 || max_T > kda::verify_max_spec_tokens()) return KDA_EINVAL;
  if (tok->num_seqs == 0) return KDA_OK;
  if (!state_slots || !snapshots) return KDA_EINVAL;
  if (!aligned16(snapshots)) return KDA_EALIGN;
  if (device_unsafe()) return KDA_EDEVICE;
  unsigned *err = device_error_word();
  if (!err) return KDA_ECUDA;
  kda::SnapshotParams p = {};
  p.q = tok->q;
  p.k = tok->k;
  p.v = tok->v;
  p.alpha = tok->alpha;
  p.beta = tok->beta;
  p.o = tok->o;
  p.cu_seqlens = tok->cu_seqlens;
  p.state_slots = state_slots;
  p.pool = pool->base;
  p.snap = snapshots;
  p.err = err;
  p.B = tok->num_seqs;
  p.N = tok->num_tokens;
  p.H = pool->num_heads;
  p.P = pool->num_slots;
  p.max_T = max_T;
  return cuda_status(kda::launch_verify_snapshot(
      p, tok->dtype, tok->d_k, reinterpret_cast<cudaStream_t>(stream)));
}

int kda_commit_snapshot(const int32_t *accepted_len, const int32_t *state_slots,
                        int32_t num_seqs, kda_state_pool *pool,
                        const float *snapshots, int32_t max_T,
                        kda_stream_t stream) {
  int st = check_pool(pool);
  if (st) return st;
  if (num_seqs < 0 || num_seqs > kMaxGridY) return KDA_EINVAL;
  if (max_T < 1 || max_T > kda::verify_max_spec_tokens()) return KDA_EINVAL;
  if (num_seqs == 0) return KDA_OK;
  if (!accepted_len || !state_slots || !snapshots) return KDA_EINVAL;
  if (!aligned16(snapshots)) return KDA_EALIGN;
  if (device_unsafe()) return KDA_EDEVICE;
  unsigned *err = device_error_word();
  if (!err) return KDA_ECUDA;
  kda::SnapshotParams p = {};
  p.accepted_len = accepted_len;
  p.state_slots = state_slots;
  p.pool = pool->base;
  p.snap = const_cast<float *>(snapshots);
  p.err = err;
  p.B = num_seqs;
  p.H = pool->num_heads;
  p.P = pool->num_slots;
  p.max_T = max_T;
  return cuda_status(kda::launch_commit_snapshot(
      p, pool->d_k, reinterpret_cast<cudaStream_t>(stream)));
}

int kda_get_device_error(int32_t *host_bits, kda_stream_t stream) {
  if (!host_bits) return KDA_EINVAL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return KDA_ECUDA;
  unsigned int bits = 0;
  if (cudaMemcpyFromSymbol(&bits, g_kda_device_error, sizeof(bits)) != cudaSuccess)
    return KDA_ECUDA;
  const unsigned int zero = 0;
  if (cudaMemcpyToSymbol(g_kda_device_error, &zero, sizeof(zero)) != cudaSuccess)
    return KDA_ECUDA;
  *host_bits = (int32_t)bits;
  if (bits & KDA_DERR_UNSAFE) {
    int dev = -1;
    if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < 64)
      g_unsafe_devices.fetch_or(1ull << dev);
  }
  return bits ? KDA_EDEVICE : KDA_OK;
}

}  // extern "C"
