// Slot-table state movement: gather pool[slots[i]] into a dense buffer, and
// copy whole slots inside a pool (prefix-cache fork of a checkpoint into a
// live slot).  Plain 128-bit streaming copies; one grid row per slot entry.
#include "kda_internal.cuh"

namespace kda {
namespace {

__global__ void slot_copy_kernel(const SlotCopyParams p) {
  const int n = blockIdx.y;
  const int s = p.src_slots[n];
  const int d = p.dst_slots ? p.dst_slots[n] : n;
  if (s < 0 || s >= p.P || (p.dst_slots && (d < 0 || d >= p.P))) {
    if (blockIdx.x == 0 && threadIdx.x == 0) set_error(p.err, KDA_DERR_SLOT);
    return;
  }
  const float4 *src = reinterpret_cast<const float4 *>(p.src_base + (size_t)s * p.state_floats);
  float4 *dst = reinterpret_cast<float4 *>(p.dst_base + (size_t)d * p.state_floats);
  const long long n4 = p.state_floats / 4;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
       i += (long long)gridDim.x * blockDim.x)
    dst[i] = src[i];
}

}  // namespace

cudaError_t launch_slot_copy(const SlotCopyParams &p, cudaStream_t s) {
  if (p.n == 0) return cudaSuccess;
  const long long n4 = p.state_floats / 4;
  int bx = (int)((n4 + 255) / 256);
  if (bx > 64) bx = 64;
  dim3 grid(bx, p.n);
  slot_copy_kernel<<<grid, 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace kda
