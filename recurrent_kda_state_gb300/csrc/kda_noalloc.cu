// Chunked prefill without a caller-provided workspace: the scratch lives in a
// fixed array of device memory owned by this library (its own translation
// unit, so only this module holds it).  The work itself is
// kda_prefill_chunked, unchanged.
#include <mutex>

#include "kda_internal.cuh"

// The scratch.  In host code this name is only a stand-in for the device
// array, never a device address: the address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char
    g_kda_noalloc_scratch[KDA_NOALLOC_SCRATCH_BYTES];

namespace {

// Device address of the scratch on the current device, looked up once per
// device (with that device current).  nullptr if the lookup failed.
unsigned char *scratch_address() {
  static std::mutex mu;
  static unsigned char *cache[64] = {};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_kda_noalloc_scratch) != cudaSuccess) return nullptr;
    cache[dev] = static_cast<unsigned char *>(p);
  }
  return cache[dev];
}

}  // namespace

extern "C" int kda_prefill_chunked_noalloc(const kda_tokens *tok,
                                           kda_state_pool *pool,
                                           const int32_t *state_slots,
                                           const int32_t *ckpt_slots,
                                           int32_t max_ckpt, int32_t ckpt_every,
                                           int32_t chunk,
                                           const int32_t *start_pos,
                                           kda_stream_t stream) {
  if (!tok || !pool) return KDA_EINVAL;
  if (tok->num_seqs == 0) return KDA_OK;
  const size_t need = kda_prefill_workspace_size(
      tok->num_tokens, tok->num_seqs, tok->num_heads, tok->d_k, tok->d_v, chunk,
      tok->dtype);
  // 0: bad arguments, which kda_prefill_chunked reports itself; at the
  // tensor-core shape a workspace larger than the scratch selects the
  // single pass, which needs none
  const bool tc = kda::prefill_uses_tc(tok->dtype, tok->num_heads, tok->d_k, tok->d_v,
                                       chunk);
  if (need == 0 || (tc && need > KDA_NOALLOC_SCRATCH_BYTES))
    return kda_prefill_chunked(tok, pool, state_slots, ckpt_slots, max_ckpt,
                               ckpt_every, chunk, start_pos, nullptr, 0, stream);
  if (need > KDA_NOALLOC_SCRATCH_BYTES) {
    // a malformed call reports what kda_prefill_chunked would, not the size
    const int st = kda::prefill_check_args(tok, pool, state_slots, ckpt_slots, max_ckpt,
                                           ckpt_every, chunk);
    return st != KDA_OK ? st : KDA_ENOSPC;
  }
  unsigned char *ws = scratch_address();
  if (!ws) return KDA_ECUDA;
  return kda_prefill_chunked(tok, pool, state_slots, ckpt_slots, max_ckpt,
                             ckpt_every, chunk, start_pos, ws,
                             KDA_NOALLOC_SCRATCH_BYTES, stream);
}
