// Chunked prefill on the tensor cores (tcgen05, accumulators in TMEM) for
// d_k = d_v = 128, chunk 64, bf16 inputs, heads a multiple of 8, with the in-pass checkpoints of
// "KDA checkpoints stay inside the prefill" (vLLM Kimi K3 optimisation page).
//
// Per chunk of C tokens with g_t = sum_{s<=t} log alpha_s (per key channel) and a
// reference row m in the middle of the chunk (every factor below stays within
// e^{+-80}, checked), with K~ = e^{g-g_m} K, Q~ = e^{g-g_m} Q, K^ = e^{-(g-g_m)} K
// and S~ = Diag(e^{g_m}) S (S the chunk-start state slice):
//   R1  G  = [K~; Q~] K^^T                         (128 x 64, K = 128)
//       A  = strict_tril(diag(beta) G_top),  M = tril(G_bottom)
//       T  = (I + A)^{-1} diag(beta)                (CUDA cores, 16x16 blocks)
//   R2  [T; M] [K~^T; V^T]^T -> W~ = T K~, U' = T V  (rows 0..63)
//   R3  [W~; Q~] S~        -> W S (rows 0..63),  Q S (rows 64..127)
//       U = U' - W S
//   R4  K^^T U            -> S' = Diag(e^{g_C}) S + Diag(e^{g_C-g_m}) K^^T U
//       [T; M] U          -> rows 64..127 accumulate M U:  O = Q S + M U
// (W = T (e^{g} K) = W~ Diag(e^{g_m}), so W S = W~ S~; the same for Q S.)
// This is the chunk (WY/UT) form of the gated delta rule with the factor
// pairs re-referenced to row m; the triangles of A and M keep it exact.
//
// Two ways to run it:
//   - prefill_tc_kernel, no workspace: one CTA per (value-column slice of NC
//     columns, head, sequence) walks the sequence's chunks and does all of
//     the above per chunk;
//   - with a workspace, prefill_tc_chunk_kernel first does everything up to
//     R2 for every (chunk, head) at once and writes the chunk's operands as
//     shared-memory images, then prefill_tc_pass_kernel walks the chunks with
//     R3, R4 and the state only (see the comment above those kernels).
// With projection-space inputs (RAW) E1 also prepares them: keys L2-
// normalised, log alpha = -softplus(z), beta = sigmoid(b).
//
// Precision: every operand that is not an exact bf16 input is split into
// bf16 hi + lo and each product runs as hi*hi + lo*hi + hi*lo (three
// kind::f16 MMAs into one fp32 accumulator, ~2^-16 relative per product; the
// chunk walk's stacked form adds lo*lo); V is an exact bf16 input and takes
// two.  The state stays fp32 in registers.
//
// Shared-memory operand tiles are 128-byte swizzled, K-major or, where the
// same bytes serve a second product transposed, read MN-major (see
// kda_umma.cuh); the TMEM accumulators sit at fixed columns.
#include <cuda.h>

#include <cstddef>
#include <mutex>

#include "kda_internal.cuh"
#include "kda_umma.cuh"

namespace kda {

namespace {

constexpr int kD = 128, kC = 64, kNC = 32, kThreads = 256;

// Byte offsets from a 1024-byte aligned base.
struct Lay {
  static constexpr uint32_t GA_HI = 0;       // [K~; Q~] then [W~; Q~]: 128 x 128
  static constexpr uint32_t GA_LO = 32768;
  static constexpr uint32_t GB_HI = 65536;   // K^: 64 x 128
  static constexpr uint32_t GB_LO = 81920;
  static constexpr uint32_t AF = 65536;      // after R1: A fp32 64 x 68
  static constexpr uint32_t XF = 82944;      //           X fp32 64 x 68
  static constexpr uint32_t UT_HI = 65536;   // after the solve: U, MN-major 64 x [hi|lo]
  static constexpr uint32_t UT_LO = UT_HI + kNC * 128;
  static constexpr uint32_t B2_HI = 101376;  // [K~^T; V^T]: (128 + NC) x 64
  static constexpr uint32_t B2_LO = B2_HI + (128 + kNC) * 128;  // K~^T lo
  static constexpr uint32_t KH_HI = B2_LO + 16384;  // K^^T: 128 x 64
  static constexpr uint32_t KH_LO = KH_HI + 16384;
  static constexpr uint32_t TM_HI = KH_LO + 16384;  // [T; M]: 128 x 64
  static constexpr uint32_t TM_LO = TM_HI + 16384;
  static constexpr uint32_t SB_HI = TM_LO + 16384;  // S~: MN-major 128 x [hi|lo]
  static constexpr uint32_t SB_LO = SB_HI + kNC * 256;
  static constexpr uint32_t MISC = SB_LO + kNC * 256;
  // misc (floats unless noted)
  static constexpr uint32_t BET = MISC;              // beta [64]
  static constexpr uint32_t GM = BET + 256;          // g_m [128]
  static constexpr uint32_t GC = GM + 512;           // g_C [128]
  static constexpr uint32_t EGC = GC + 512;          // e^{g_C} [128]
  static constexpr uint32_t ECM = EGC + 512;         // e^{g_C - g_m} [128]
  static constexpr uint32_t PT = ECM + 512;          // solve blocks 3 x 256
  static constexpr uint32_t TOT4 = PT + 3072;        // quarter sums [4][128]
  static constexpr uint32_t BST = TOT4 + 2048;       // staged beta bf16 [64][8]
  static constexpr uint32_t MBAR = BST + 1024;       // u64: tensor cores
  static constexpr uint32_t SBAR = MBAR + 8;         // u64: staging copies
  static constexpr uint32_t TSLOT = SBAR + 8;        // u32
  static constexpr uint32_t END = TSLOT + 8;
  static constexpr size_t kBytes = END + 1024;       // + alignment slack
};
static_assert(Lay::B2_LO % 1024 == 0 && Lay::KH_HI % 1024 == 0 &&
                  Lay::SB_HI % 1024 == 0 && Lay::UT_LO % 1024 == 0,
              "tiles on 1024-byte boundaries");
static_assert(Lay::UT_LO + kNC * 128 <= Lay::B2_HI, "U^T fits the K^ region");
static_assert(Lay::XF + 64 * 68 * 4 <= Lay::B2_HI && Lay::XF >= Lay::AF + 64 * 68 * 4,
              "A and X fit before the R2 B tile");
// The next chunk's raw rows are staged while this chunk's R3/R4 run, in
// regions free from the end of R2 to the next E1: q, k (bf16 [64][128]) in
// the R2 B tile, alpha in the X array, the V slice after U^T.
constexpr uint32_t kStgQ = Lay::B2_HI, kStgK = Lay::B2_HI + 16384;
constexpr uint32_t kStgA = Lay::XF, kStgV = Lay::UT_LO + kNC * 128;
static_assert(kStgK + 16384 <= Lay::B2_HI + (128 + kNC) * 128 + 16384, "q, k staging");
static_assert(kStgV + 64 * kNC * 2 <= Lay::XF, "V staging");
static_assert(Lay::kBytes <= 232448, "shared memory per CTA");

// TMEM columns of the accumulators (512 allocated).
// R3 and R4 take the hi and lo splits of their B operand stacked along N
// (N = 64): columns 0..31 of kAcc3 / kAcc4 hold hi*hi + lo*hi, 32..63 hi*lo +
// lo*lo, and a result is their sum.
constexpr uint32_t kAccG = 0, kAcc2 = 64, kAcc3 = 64 + 128 + kNC,
                   kAcc4 = kAcc3 + 2 * kNC;
static_assert(kAcc4 + 2 * kNC <= 512, "TMEM columns");

// Index of element (r, c) of a 64 x 64 fp32 array with rows 68 floats apart:
// rows stay 16-byte aligned and a column's 8 consecutive rows fall in
// distinct banks.
__device__ __forceinline__ int fo(int r, int c) { return r * 68 + c; }

__device__ __forceinline__ void st_v4(uint8_t *base, uint32_t off, uint32_t a,
                                      uint32_t b, uint32_t c, uint32_t d) {
  *reinterpret_cast<uint4 *>(base + off) = make_uint4(a, b, c, d);
}

// Eight fp32 values -> one 16-byte chunk of a hi tile and of a lo tile.
__device__ __forceinline__ void put8(uint8_t *sm, uint32_t hi_off, uint32_t lo_off,
                                     const float *x) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) umma::split_bf16x2(x[2 * i], x[2 * i + 1], h[i], l[i]);
  st_v4(sm, hi_off, h[0], h[1], h[2], h[3]);
  st_v4(sm, lo_off, l[0], l[1], l[2], l[3]);
}

// Sixteen fp32 values x[0..15] of K-row k, MN positions n0 .. n0 + 15 (n0 a
// multiple of 16, < 32) -> an MN-major tile holding the hi split at n and the
// lo split at 32 + n: four 16-byte chunks.
__device__ __forceinline__ void put16_mn(uint8_t *sm, uint32_t tile, int k, int n0,
                                         const float *x) {
  uint32_t h[8], l[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) umma::split_bf16x2(x[2 * i], x[2 * i + 1], h[i], l[i]);
  st_v4(sm, tile + umma::sw128_mn_off16(k, n0), h[0], h[1], h[2], h[3]);
  st_v4(sm, tile + umma::sw128_mn_off16(k, n0 + 8), h[4], h[5], h[6], h[7]);
  st_v4(sm, tile + umma::sw128_mn_off16(k, kNC + n0), l[0], l[1], l[2], l[3]);
  st_v4(sm, tile + umma::sw128_mn_off16(k, kNC + n0 + 8), l[4], l[5], l[6], l[7]);
}

// Four consecutive entries (r, c..c+3) of a swizzled 64 x 64 fp32 array
// (c a multiple of 4).
__device__ __forceinline__ float4 ld4(const float *M, int r, int c) {
  return *reinterpret_cast<const float4 *>(M + fo(r, c));
}

// One block distance d of the off-diagonal pass: for the 4 - d blocks
// (a, b) = (blk + d, blk), P_ab = sum_{b<=r<a} A_ar X_rb (16 x 16 each).
// Thread -> row i and four columns j0..j0+3 of one block (threads past the
// 64 (4 - d) strips idle); X rows and A rows are read as float4.
template <int d>
__device__ __forceinline__ void offdiag_sum(const float *A, const float *X,
                                            float *P, int tid) {
  if (tid < 64 * (4 - d)) {
    const int blk = tid >> 6, i = (tid >> 2) & 15, j0 = (tid & 3) * 4;
    const int a = blk + d, b = blk;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int rr = 0; rr < d; ++rr) {
      const int rb = b + rr;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float4 av = ld4(A, 16 * a + i, 16 * rb + 4 * k);
        const float aw[4] = {av.x, av.y, av.z, av.w};
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const float4 x = ld4(X, 16 * rb + 4 * k + m, 16 * b + j0);
          acc.x = fmaf(aw[m], x.x, acc.x);
          acc.y = fmaf(aw[m], x.y, acc.y);
          acc.z = fmaf(aw[m], x.z, acc.z);
          acc.w = fmaf(aw[m], x.w, acc.w);
        }
      }
    }
    *reinterpret_cast<float4 *>(P + blk * 256 + i * 16 + j0) = acc;
  }
}

// X_ab = -X_aa P_ab for the blocks of distance d (same thread mapping).
template <int d>
__device__ __forceinline__ void offdiag_apply(const float *P, float *X, int tid) {
  if (tid < 64 * (4 - d)) {
    const int blk = tid >> 6, i = (tid >> 2) & 15, j0 = (tid & 3) * 4;
    const int a = blk + d, b = blk;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float4 xv = ld4(X, 16 * a + i, 16 * a + 4 * k);
      const float xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const float4 pv = *reinterpret_cast<const float4 *>(P + blk * 256 + (4 * k + m) * 16 + j0);
        acc.x = fmaf(xw[m], pv.x, acc.x);
        acc.y = fmaf(xw[m], pv.y, acc.y);
        acc.z = fmaf(xw[m], pv.z, acc.z);
        acc.w = fmaf(xw[m], pv.w, acc.w);
      }
    }
    *reinterpret_cast<float4 *>(X + fo(16 * a + i, 16 * b + j0)) =
        make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
  }
}

// X = (I + A)^{-1} for a strictly lower-triangular 64 x 64 A (fp32 arrays,
// row stride 68), by 16 x 16 blocks: diagonal blocks by forward substitution (one
// column per thread, each row of A read as four float4), then
// X_ab = -X_aa sum_{b<=r<a} A_ar X_rb by block distance a - b = 1, 2, 3.
// X's strictly upper part is not written.
__device__ void unit_lower_inverse(const float *A, float *X, float *P, int tid) {
  if (tid < 64) {
    const int o = (tid >> 4) * 16, j = tid & 15;
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float4 av[4];
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (4 * k < i) av[k] = ld4(A, o + i, o + 4 * k);
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int r = 0; r < i; ++r) {
        const float4 v = av[r >> 2];
        const float arr = (r & 3) == 0 ? v.x : (r & 3) == 1 ? v.y : (r & 3) == 2 ? v.z : v.w;
        acc[r & 3] = fmaf(arr, x[r], acc[r & 3]);
      }
      const float sum = (acc[0] + acc[1]) + (acc[2] + acc[3]);
      x[i] = i < j ? 0.f : (i == j ? 1.f : -sum);
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) X[fo(o + i, o + j)] = x[i];
  }
  __syncthreads();
  offdiag_sum<1>(A, X, P, tid);
  __syncthreads();
  offdiag_apply<1>(P, X, tid);
  __syncthreads();
  offdiag_sum<2>(A, X, P, tid);
  __syncthreads();
  offdiag_apply<2>(P, X, tid);
  __syncthreads();
  offdiag_sum<3>(A, X, P, tid);
  __syncthreads();
  offdiag_apply<3>(P, X, tid);
  __syncthreads();
}

// Input prep for projection-space inputs (the generator's formulas; the
// pages leave it open): log alpha = -softplus(z), beta = sigmoid(b), and the
// key's inverse L2 norm over the 128 channels of one (token, head).
__device__ __forceinline__ float neg_softplus(float z) {
  return -(fmaxf(z, 0.f) + __logf(1.f + __expf(-fabsf(z))));
}
__device__ __forceinline__ float sigmoid_f(float b) {
  return __fdividef(1.f, 1.f + __expf(-b));
}
// E1 thread (channel pair cp, token quarter tq) holding bf16 key pairs kr[u]
// of tokens 16 tq + u: per-token sums of squares over the 64 channel pairs
// (two warps per quarter) -> scr[warp][u]; after a barrier, norm_finish
// turns them into inverse norms nrm[t] (threads cp == 0).
__device__ __forceinline__ void norm_partials(const uint32_t (&kr)[16], float *scr, int tid) {
#pragma unroll
  for (int u = 0; u < 16; ++u) {
    const float k0 = __uint_as_float(kr[u] << 16), k1 = __uint_as_float(kr[u] & 0xffff0000u);
    float x = fmaf(k0, k0, k1 * k1);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    if ((tid & 31) == 0) scr[(tid >> 5) * 16 + u] = x;
  }
}
__device__ __forceinline__ void norm_finish(const float *scr, float *nrm, int tid) {
  if ((tid & 63) == 0) {
    const int tq = tid >> 6;
#pragma unroll
    for (int u = 0; u < 16; ++u)
      nrm[16 * tq + u] = rsqrtf(fmaxf(scr[(2 * tq) * 16 + u] + scr[(2 * tq + 1) * 16 + u],
                                      1e-24f));
  }
}

// Descriptor of a tile `off` bytes past the one `d` describes (the start
// address field counts 16-byte units).
__device__ __forceinline__ uint64_t dadd(uint64_t d, uint32_t off) {
  return d + (off >> 4);
}

// Every thread waits for the barrier's phase (bounded); they agree whether
// it completed.  On success the phase advances.
__device__ __forceinline__ bool tc_wait(uint64_t *mbar, uint32_t &phase, int limit) {
  const bool ok = umma::mbar_wait(mbar, phase, limit);
  const bool all = __syncthreads_and(ok) != 0;
  if (all) phase ^= 1u;
  umma::fence_after_sync();
  return all;
}

// This thread waits for the barrier's phase (bounded) with no block barrier:
// the caller folds the outcome into the next barrier it crosses
// (tiles_ready_and / __syncthreads_and), so every thread still agrees before
// acting on it.  On success the phase advances.
__device__ __forceinline__ bool own_wait(uint64_t *mbar, uint32_t &phase, int limit) {
  const bool ok = umma::mbar_wait(mbar, phase, limit);
  if (ok) phase ^= 1u;
  umma::fence_after_sync();
  return ok;
}

// Publish this thread's shared-memory tile writes to the tensor core and
// meet the MMA-issuing thread.
__device__ __forceinline__ void tiles_ready() {
  umma::fence_smem_to_async();
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
}
// tiles_ready() that also agrees on every thread's `ok`.
__device__ __forceinline__ bool tiles_ready_and(bool ok) {
  umma::fence_smem_to_async();
  umma::fence_before_sync();
  const bool all = __syncthreads_and(ok) != 0;
  umma::fence_after_sync();
  return all;
}

// Tensor maps of the packed inputs viewed as [N][H][D] (3-D, innermost D):
// boxes of 64 tokens x 1 head x 128 channels (q, k, alpha) or x NC channels
// (v); rows past N read as zeros.
struct InputMaps {
  CUtensorMap q, k, a, v, b;  // b: beta [N][H] as 2-D, boxes of 8 heads x 64 tokens
};
static_assert(offsetof(InputMaps, b) == offsetof(InputMaps, q) + 4 * sizeof(CUtensorMap),
              "the five maps are consecutive");

// Threads 32 .. 36 prefetch the five maps' descriptors, which a copy would
// otherwise fetch at its first use.
__device__ __forceinline__ void prefetch_input_maps(const InputMaps &maps, int tid) {
  if (tid >= 32 && tid < 37)
    asm volatile("prefetch.tensormap [%0];"
                 :: "l"(reinterpret_cast<uint64_t>(&maps.q + (tid - 32))) : "memory");
}

// One TMA load of a 2-D box of `tm` at (x, token) into shared memory,
// completing its bytes on the mbarrier's transaction count.
__device__ __forceinline__ void tma_load2(uint32_t dst, const CUtensorMap *tm, int x,
                                          int tok, uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];"
      :: "r"(dst), "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(tok), "r"(mbar)
      : "memory");
}

// One TMA load of a box of `tm` at (x, head, token) into shared memory,
// completing its bytes on the mbarrier's transaction count.
__device__ __forceinline__ void tma_load3(uint32_t dst, const CUtensorMap *tm, int x,
                                          int head, int tok, uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];"
      :: "r"(dst), "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(head), "r"(tok),
         "r"(mbar) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t mbar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
               :: "r"(mbar), "r"(bytes) : "memory");
}


template <bool RAW>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const PrefillParams p, const __grid_constant__ InputMaps maps) {
  extern __shared__ float4 smem4[];
  uint8_t *sm = umma::align1024(smem4);
  const uint32_t sb = umma::smem_u32(sm);
  float *bet = reinterpret_cast<float *>(sm + Lay::BET);
  float *sgm = reinterpret_cast<float *>(sm + Lay::GM);
  float *sgc = reinterpret_cast<float *>(sm + Lay::GC);
  float *tot4 = reinterpret_cast<float *>(sm + Lay::TOT4);
  float *egc = reinterpret_cast<float *>(sm + Lay::EGC);
  float *ecm = reinterpret_cast<float *>(sm + Lay::ECM);
  float *Af = reinterpret_cast<float *>(sm + Lay::AF);
  float *Xf = reinterpret_cast<float *>(sm + Lay::XF);
  uint64_t *mbar = reinterpret_cast<uint64_t *>(sm + Lay::MBAR);
  uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + Lay::TSLOT);
  prefetch_input_maps(maps, threadIdx.x);

  const int tid = threadIdx.x, sl = blockIdx.x, h = blockIdx.y, i = blockIdx.z;
  const int H = p.H, col0 = sl * kNC;
  const int c = tid & 127, hf = tid >> 7;  // key channel = TMEM lane; half

  const int cu0 = p.cu_seqlens[i], cu1 = p.cu_seqlens[i + 1];
  const int L = cu1 - cu0;
  const int p0 = p.start_pos ? p.start_pos[i] : 0;
  if (cu0 < 0 || L < 0 || cu1 > p.N || p0 < 0) {
    if (tid == 0 && sl == 0) set_error(p.err, KDA_DERR_SEGMENT);
    return;
  }
  if (L == 0) return;
  const int slot = p.state_slots[i];
  if (slot < 0 || slot >= p.P) {
    if (tid == 0 && sl == 0) set_error(p.err, KDA_DERR_SLOT);
    return;
  }

  if (tid < 32) umma::tmem_alloc(tslot, 512);
  if (tid == 0) {
    umma::mbar_init(mbar, 1);
    umma::mbar_init(reinterpret_cast<uint64_t *>(sm + Lay::SBAR), 1);
  }
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tmem = *tslot;
  const uint32_t tl = tmem + ((uint32_t)(tid & 96) << 16);  // lane quadrant
  uint32_t phase = 0;
  const uint32_t sbar = sb + Lay::SBAR;
  const uint64_t dGA = umma::sdesc_sw128(sb + Lay::GA_HI);  // all tiles from here
  uint32_t sphase = 0;        // next phase of the staging barrier
  bool stage_owed = false;    // copies issued and not yet waited for

  // S[c][col0 + 16 hf + jj], fp32, for the whole pass
  float S[16];
  {
    const float *src = p.pool + ((size_t)slot * H + h) * kD * kD;
#pragma unroll
    for (int jj = 0; jj < 16; ++jj)
      S[jj] = src[(size_t)(col0 + 16 * hf + jj) * kD + c];
  }

  const int r0 = p0 % kC;
  const int nch = (r0 + L + kC - 1) / kC;
  // TMA loads of chunk qq's 64 rows of q, k, alpha, the V slice and beta
  // (the 8 heads around h) into the staging areas (rows past the chunk are
  // masked where they are read), completing on the staging barrier.
  auto stage = [&](int qq) {
    const int s0 = max(0, qq * kC - r0);
    if (tid == 0) {
      mbar_expect_tx(sbar, 3 * 64 * 2 * kD + 64 * 2 * kNC + 64 * 16);
      tma_load3(sb + kStgQ, &maps.q, 0, h, cu0 + s0, sbar);
      tma_load3(sb + kStgK, &maps.k, 0, h, cu0 + s0, sbar);
      tma_load3(sb + kStgA, &maps.a, 0, h, cu0 + s0, sbar);
      tma_load3(sb + kStgV, &maps.v, col0, h, cu0 + s0, sbar);
      tma_load2(sb + Lay::BST, &maps.b, h & ~7, cu0 + s0, sbar);
    }
    stage_owed = true;
  };
  stage(0);
  bool ok = true, mma_owed = false;  // an MMA round in flight
  for (int q = 0; q < nch; ++q) {
    const int s_loc = max(0, q * kC - r0);
    const int e_loc = min(L, (q + 1) * kC - r0);
    const int n = e_loc - s_loc, tok0 = cu0 + s_loc, m = n >> 1;

    // ---- E1: the chunk's raw rows are in the staging areas.  Thread
    // (channel pair cp, token quarter tq) takes channels 2cp, 2cp+1 of rows
    // 16tq .. 16tq+15: cumulative log-decay (padded rows: alpha = 1), then the
    // scaled operand tiles; S~ from the state rows this thread owns.
    if (!(ok = tc_wait(reinterpret_cast<uint64_t *>(sm + Lay::SBAR), sphase, p.spin_limit))) break;
    stage_owed = false;
    if (tid < kC) {
      const uint16_t bw = reinterpret_cast<const uint16_t *>(sm + Lay::BST)[tid * 8 + (h & 7)];
      const float bv = __uint_as_float((uint32_t)bw << 16);
      bet[tid] = tid < n ? (RAW ? sigmoid_f(bv) : bv) : 0.f;
    }
    const int cp = tid & 63, tq = tid >> 6, c2 = 2 * cp, tb0 = 16 * tq;
    float la0[16], la1[16];
    uint32_t kr[16], qr[16];
    {
      const uint32_t *sq = reinterpret_cast<const uint32_t *>(sm + kStgQ);
      const uint32_t *sk = reinterpret_cast<const uint32_t *>(sm + kStgK);
      const uint32_t *sa = reinterpret_cast<const uint32_t *>(sm + kStgA);
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int t = tb0 + u;
        const uint32_t aw = sa[t * 64 + cp];
        kr[u] = t < n ? sk[t * 64 + cp] : 0u;
        qr[u] = t < n ? sq[t * 64 + cp] : 0u;
        const float a0 = __uint_as_float(aw << 16), a1 = __uint_as_float(aw & 0xffff0000u);
        la0[u] = t < n ? (RAW ? neg_softplus(a0) : __logf(a0)) : 0.f;
        la1[u] = t < n ? (RAW ? neg_softplus(a1) : __logf(a1)) : 0.f;
      }
    }
    float *nscr = reinterpret_cast<float *>(sm + Lay::PT);   // key norms (raw inputs)
    float *nrm = nscr + 128;
    if (RAW) norm_partials(kr, nscr, tid);
    uint32_t vw[4];
    {
      const int j = tid & 31, tg = tid >> 5;
      const uint16_t *vs = reinterpret_cast<const uint16_t *>(sm + kStgV);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int ta = 8 * tg + 2 * e;
        vw[e] = (ta < n ? (uint32_t)vs[ta * kNC + j] : 0u) |
                (ta + 1 < n ? (uint32_t)vs[(ta + 1) * kNC + j] << 16 : 0u);
      }
    }
#pragma unroll
    for (int u = 1; u < 16; ++u) {
      la0[u] += la0[u - 1];
      la1[u] += la1[u - 1];
    }
    tot4[tq * 128 + c2] = la0[15];
    tot4[tq * 128 + c2 + 1] = la1[15];
    __syncthreads();  // staging consumed; quarter sums visible
    {
      float add0 = 0.f, add1 = 0.f;
      for (int w = 0; w < tq; ++w) {
        add0 += tot4[w * 128 + c2];
        add1 += tot4[w * 128 + c2 + 1];
      }
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        la0[u] += add0;
        la1[u] += add1;
        if (tb0 + u == m) {
          sgm[c2] = la0[u];
          sgm[c2 + 1] = la1[u];
        }
      }
      if (tq == 3) {
        sgc[c2] = la0[15];
        sgc[c2 + 1] = la1[15];
      }
    }
    if (RAW) norm_finish(nscr, nrm, tid);
    __syncthreads();
    {
      const float gm0 = sgm[c2], gm1 = sgm[c2 + 1];
      if (tq == 0) {
        const float gC0 = sgc[c2], gC1 = sgc[c2 + 1];
        if (la0[0] - gm0 > 80.f || gm0 - gC0 > 80.f || la1[0] - gm1 > 80.f ||
            gm1 - gC1 > 80.f)
          set_error(p.err, KDA_DERR_RANGE);
        egc[c2] = __expf(gC0);
        egc[c2 + 1] = __expf(gC1);
        ecm[c2] = __expf(gC0 - gm0);
        ecm[c2 + 1] = __expf(gC1 - gm1);
      }
      // bf16 halves of K~ and K^ for channels (c2, c2 + 1) of the last 8
      // rows: the transposed tiles take them as they are (byte permutes)
      uint32_t ktH[8], ktL[8], khH[8], khL[8];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int t = tb0 + u;
        const float f0 = __expf(la0[u] - gm0), fi0 = __expf(gm0 - la0[u]);
        const float f1 = __expf(la1[u] - gm1), fi1 = __expf(gm1 - la1[u]);
        const float kn = RAW ? nrm[t] : 1.f;
        const float k0 = __uint_as_float(kr[u] << 16) * kn;
        const float k1 = __uint_as_float(kr[u] & 0xffff0000u) * kn;
        const float q0 = __uint_as_float(qr[u] << 16);
        const float q1 = __uint_as_float(qr[u] & 0xffff0000u);
        uint32_t hi, lo;
        uint32_t off = umma::sw128_off16(t, c2, 128);
        umma::split_bf16x2(f0 * k0, f1 * k1, ktH[u & 7], ktL[u & 7]);
        *reinterpret_cast<uint32_t *>(sm + Lay::GA_HI + off) = ktH[u & 7];
        *reinterpret_cast<uint32_t *>(sm + Lay::GA_LO + off) = ktL[u & 7];
        off = umma::sw128_off16(64 + t, c2, 128);
        umma::split_bf16x2(f0 * q0, f1 * q1, hi, lo);
        *reinterpret_cast<uint32_t *>(sm + Lay::GA_HI + off) = hi;
        *reinterpret_cast<uint32_t *>(sm + Lay::GA_LO + off) = lo;
        off = umma::sw128_off16(t, c2, 64);
        umma::split_bf16x2(fi0 * k0, fi1 * k1, khH[u & 7], khL[u & 7]);
        *reinterpret_cast<uint32_t *>(sm + Lay::GB_HI + off) = khH[u & 7];
        *reinterpret_cast<uint32_t *>(sm + Lay::GB_LO + off) = khL[u & 7];
        if ((u & 7) == 7) {
          const int tb = t - 7;
#pragma unroll
          for (int e = 0; e < 2; ++e) {  // row c2 + e: low (e = 0) or high halves
            const uint32_t sel = e ? 0x7632u : 0x5410u;
            const int row = c2 + e;
            st_v4(sm, Lay::B2_HI + umma::sw128_off16(row, tb, 128 + kNC),
                  __byte_perm(ktH[0], ktH[1], sel), __byte_perm(ktH[2], ktH[3], sel),
                  __byte_perm(ktH[4], ktH[5], sel), __byte_perm(ktH[6], ktH[7], sel));
            st_v4(sm, Lay::B2_LO + umma::sw128_off16(row, tb, 128),
                  __byte_perm(ktL[0], ktL[1], sel), __byte_perm(ktL[2], ktL[3], sel),
                  __byte_perm(ktL[4], ktL[5], sel), __byte_perm(ktL[6], ktL[7], sel));
            st_v4(sm, Lay::KH_HI + umma::sw128_off16(row, tb, 128),
                  __byte_perm(khH[0], khH[1], sel), __byte_perm(khH[2], khH[3], sel),
                  __byte_perm(khH[4], khH[5], sel), __byte_perm(khH[6], khH[7], sel));
            st_v4(sm, Lay::KH_LO + umma::sw128_off16(row, tb, 128),
                  __byte_perm(khL[0], khL[1], sel), __byte_perm(khL[2], khL[3], sel),
                  __byte_perm(khL[4], khL[5], sel), __byte_perm(khL[6], khL[7], sel));
          }
        }
      }
    }
    {
      const float egm = __expf(sgm[c]);
      float x[16];
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) x[jj] = egm * S[jj];
      put16_mn(sm, Lay::SB_HI, c, 16 * hf, x);  // MN-major, hi and lo stacked
    }
    {  // V^T rows of the R2 B tile: exact bf16, hi part only
      const int j = tid & 31, tg = tid >> 5;
      st_v4(sm, Lay::B2_HI + umma::sw128_off16(128 + j, 8 * tg, 128 + kNC), vw[0],
            vw[1], vw[2], vw[3]);
    }
    tiles_ready();

    // ---- R1: G = [K~; Q~] K^^T
    if (tid == 0) {
      const uint32_t id = umma::idesc_bf16(128, 64);
      for (int ps = 0; ps < 3; ++ps) {
        const uint32_t a = ps == 1 ? Lay::GA_LO : Lay::GA_HI;
        const uint32_t b = ps == 2 ? Lay::GB_LO : Lay::GB_HI;
        for (int kk = 0; kk < 8; ++kk)
          umma::mma_bf16(tmem + kAccG, dadd(dGA, a + (kk >> 2) * 16384 + (kk & 3) * 32),
                         dadd(dGA, b + (kk >> 2) * 8192 + (kk & 3) * 32), id,
                         (uint32_t)(ps | kk));
      }
      umma::commit(mbar);
    }
    mma_owed = true;
    if (!(ok = tc_wait(mbar, phase, p.spin_limit))) break;
    mma_owed = false;
    {  // A = strict_tril(diag(beta) G_top) -> fp32;  M = tril(G_bottom) -> tile
      float g[32];
      {
        float g0[16], g1[16];
        umma::tmem_ld16(tl + kAccG + 32 * hf, g0);
        umma::tmem_ld16(tl + kAccG + 32 * hf + 16, g1);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          g[e] = g0[e];
          g[16 + e] = g1[e];
        }
      }
      if (c < 64) {
        const int t = c;
        const float bt = bet[t];
#pragma unroll
        for (int s4 = 0; s4 < 8; ++s4) {
          const int s = 32 * hf + 4 * s4;
          float4 v;
          v.x = s < t ? bt * g[4 * s4] : 0.f;
          v.y = s + 1 < t ? bt * g[4 * s4 + 1] : 0.f;
          v.z = s + 2 < t ? bt * g[4 * s4 + 2] : 0.f;
          v.w = s + 3 < t ? bt * g[4 * s4 + 3] : 0.f;
          *reinterpret_cast<float4 *>(Af + fo(t, s)) = v;
        }
      } else {
        const int t = c - 64;
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          const int s = 32 * hf + 8 * ch;
          float x[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] = s + e <= t ? g[8 * ch + e] : 0.f;
          put8(sm, Lay::TM_HI + umma::sw128_off16(64 + t, s, 128),
               Lay::TM_LO + umma::sw128_off16(64 + t, s, 128), x);
        }
      }
    }
    __syncthreads();
    unit_lower_inverse(Af, Xf, reinterpret_cast<float *>(sm + Lay::PT), tid);
    {  // T = X diag(beta) -> rows 0..63 of the [T; M] tile
      const int t = tid >> 2, s0 = (tid & 3) * 16;
      float x[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int s = s0 + e;
        x[e] = s <= t ? Xf[fo(t, s)] * bet[s] : 0.f;
      }
      put8(sm, Lay::TM_HI + umma::sw128_off16(t, s0, 128),
           Lay::TM_LO + umma::sw128_off16(t, s0, 128), x);
      put8(sm, Lay::TM_HI + umma::sw128_off16(t, s0 + 8, 128),
           Lay::TM_LO + umma::sw128_off16(t, s0 + 8, 128), x + 8);
    }
    tiles_ready();

    // ---- R2: [T; M] [K~^T; V^T]^T -> rows 0..63: W~ (cols 0..127), U' (128..)
    if (tid == 0) {
      for (int ps = 0; ps < 3; ++ps) {
        const uint32_t a = ps == 1 ? Lay::TM_LO : Lay::TM_HI;
        const uint32_t b = ps == 2 ? Lay::B2_LO : Lay::B2_HI;
        const uint32_t id = umma::idesc_bf16(128, ps == 2 ? 128 : 128 + kNC);
        for (int kk = 0; kk < 4; ++kk)
          umma::mma_bf16(tmem + kAcc2, dadd(dGA, a + kk * 32), dadd(dGA, b + kk * 32), id,
                         (uint32_t)(ps | kk));
      }
      umma::commit(mbar);
    }
    mma_owed = true;
    if (!(ok = tc_wait(mbar, phase, p.spin_limit))) break;
    mma_owed = false;
    if (q + 1 < nch) stage(q + 1);  // the R2 B tile and X are free now
    float up[16];
    if (c < 64) {  // W~ row t -> rows 0..63 of the R3 A tile; U' kept
      const int t = c;
#pragma unroll
      for (int blk = 0; blk < 4; ++blk) {
        float w[16];
        const int k0 = 64 * hf + 16 * blk;
        umma::tmem_ld16(tl + kAcc2 + k0, w);
        put8(sm, Lay::GA_HI + umma::sw128_off16(t, k0, 128),
             Lay::GA_LO + umma::sw128_off16(t, k0, 128), w);
        put8(sm, Lay::GA_HI + umma::sw128_off16(t, k0 + 8, 128),
             Lay::GA_LO + umma::sw128_off16(t, k0 + 8, 128), w + 8);
      }
      umma::tmem_ld16(tl + kAcc2 + 128 + 16 * hf, up);
    }
    tiles_ready();

    // ---- R3: [W~; Q~] S~ -> W S (rows 0..63), Q S (rows 64..127)
    if (tid == 0) {  // A_hi [S~_hi | S~_lo], then A_lo [S~_hi | S~_lo] (N = 64)
      const uint32_t id = umma::idesc_bf16_bmn(128, 2 * kNC);
      const uint64_t dSB = umma::sdesc_sw128_mn(sb + Lay::SB_HI);
      for (int ps = 0; ps < 2; ++ps) {
        const uint32_t a = ps ? Lay::GA_LO : Lay::GA_HI;
        for (int kk = 0; kk < 8; ++kk)
          umma::mma_bf16(tmem + kAcc3, dadd(dGA, a + (kk >> 2) * 16384 + (kk & 3) * 32),
                         dadd(dSB, kk * 2048), id, (uint32_t)(ps | kk));
      }
      umma::commit(mbar);
    }
    mma_owed = true;
    if (!(ok = tc_wait(mbar, phase, p.spin_limit))) break;
    mma_owed = false;
    if (c < 64) {  // U = U' - W S -> U^T tile (row j, k = t)
      const int t = c;
      float ws[16], ws2[16];
      umma::tmem_ld16(tl + kAcc3 + 16 * hf, ws);
      umma::tmem_ld16(tl + kAcc3 + kNC + 16 * hf, ws2);
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) ws[jj] = up[jj] - (ws[jj] + ws2[jj]);
      put16_mn(sm, Lay::UT_HI, t, 16 * hf, ws);  // MN-major, hi and lo stacked
    }
    tiles_ready();

    // ---- R4: K^^T U -> state increment; [T; M] U accumulates M U on Q S
    if (tid == 0) {  // both A splits against [U_hi | U_lo] (N = 64)
      const uint32_t id = umma::idesc_bf16_bmn(128, 2 * kNC);
      const uint64_t dUT = umma::sdesc_sw128_mn(sb + Lay::UT_HI);
      for (int ps = 0; ps < 2; ++ps) {
        const uint32_t a = ps ? Lay::KH_LO : Lay::KH_HI;
        for (int kk = 0; kk < 4; ++kk)
          umma::mma_bf16(tmem + kAcc4, dadd(dGA, a + kk * 32), dadd(dUT, kk * 2048), id,
                         (uint32_t)(ps | kk));
      }
      for (int ps = 0; ps < 2; ++ps) {
        const uint32_t a = ps ? Lay::TM_LO : Lay::TM_HI;
        for (int kk = 0; kk < 4; ++kk)
          umma::mma_bf16(tmem + kAcc3, dadd(dGA, a + kk * 32), dadd(dUT, kk * 2048), id, 1u);
      }
      umma::commit(mbar);
    }
    mma_owed = true;
    if (!(ok = tc_wait(mbar, phase, p.spin_limit))) break;
    mma_owed = false;
    {
      float acc[16], acc2[16];
      umma::tmem_ld16(tl + kAcc4 + 16 * hf, acc);
      umma::tmem_ld16(tl + kAcc4 + kNC + 16 * hf, acc2);
      const float a1 = egc[c], a2 = ecm[c];
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) S[jj] = fmaf(a1, S[jj], a2 * (acc[jj] + acc2[jj]));
      if (c >= 64) {  // outputs of row t = c - 64
        float o[16], o2[16];
        umma::tmem_ld16(tl + kAcc3 + 16 * hf, o);
        umma::tmem_ld16(tl + kAcc3 + kNC + 16 * hf, o2);
        const int t = c - 64;
        if (t < n) {
          float4 *dst = reinterpret_cast<float4 *>(
              p.o + ((size_t)(tok0 + t) * H + h) * kD + col0 + 16 * hf);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            dst[e] = make_float4(o[4 * e] + o2[4 * e], o[4 * e + 1] + o2[4 * e + 1],
                                 o[4 * e + 2] + o2[4 * e + 2], o[4 * e + 3] + o2[4 * e + 3]);
        }
      }
    }
    // in-pass checkpoint at an absolute block boundary
    const int P_end = p0 + e_loc;
    if (p.ckpt_every > 0 && P_end % p.ckpt_every == 0 && p.ckpt_slots) {
      const int mth = P_end / p.ckpt_every - p0 / p.ckpt_every - 1;
      if (mth >= 0 && mth < p.max_ckpt) {
        const int cs = p.ckpt_slots[(size_t)i * p.max_ckpt + mth];
        if (cs >= p.P) {
          if (tid == 0 && sl == 0) set_error(p.err, KDA_DERR_SLOT);
        } else if (cs >= 0) {
          float *dst = p.pool + ((size_t)cs * H + h) * kD * kD;
#pragma unroll
          for (int jj = 0; jj < 16; ++jj)
            dst[(size_t)(col0 + 16 * hf + jj) * kD + c] = S[jj];
        }
      }
    }
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
  }
  if (!ok) {
    if (tid == 0) {
      set_error(p.err, KDA_DERR_TIMEOUT);
      // one more bounded chance for the tensor cores before TMEM is freed
      if (mma_owed && !umma::mbar_wait(mbar, phase, kDrainWaitPolls))
        set_error(p.err, KDA_DERR_UNSAFE);
    }
  } else {
    float *dst = p.pool + ((size_t)slot * H + h) * kD * kD;
#pragma unroll
    for (int jj = 0; jj < 16; ++jj) dst[(size_t)(col0 + 16 * hf + jj) * kD + c] = S[jj];
  }
  // no copy into shared memory outlives the CTA
  if (stage_owed && tid == 0)
    if (!umma::mbar_wait(reinterpret_cast<uint64_t *>(sm + Lay::SBAR), sphase, kDrainWaitPolls))
      set_error(p.err, KDA_DERR_UNSAFE);
  umma::fence_before_sync();
  __syncthreads();
  if (tid < 32) umma::tmem_dealloc(tmem, 512);
}


// ---------------------------------------------------------------------------
// Two passes through a workspace.  The fused kernel above spends most of a
// chunk on work that does not depend on the state (E1, R1, the inverse, R2)
// inside the sequential chunk chain, and repeats it in each value slice.
// With a workspace that work runs once per (chunk, head), for all chunks at
// once, and the chain keeps R3, R4 and the state update:
//   pass 1, prefill_tc_chunk_kernel: two persistent CTAs per SM walk the
//     (chunk, head) items: E1, R1, the inverse and R2 as above with R2 over
//     all 128 value columns, and the chunk's workspace entry: the [W~; Q~],
//     K^^T and [T; M] tiles as the shared-memory images the MMAs read (bf16
//     hi/lo, 128B-swizzled, 1024-byte aligned, so a bulk copy restores the
//     swizzle), U' as fp32 in four 32-column slices, and e^{g_m}, e^{g_C},
//     e^{g_C - g_m}.  Each part of the entry is stored from registers as soon
//     as it is computed, so a CTA keeps only the operands of its own MMAs in
//     shared memory (about 100 KB) and two items share an SM: one's CUDA-core
//     phases run while the other waits on its MMAs or its loads;
//   pass 2, prefill_tc_pass_kernel: one CTA per (value slice, head, sequence)
//     walks the chunks: S~ tile, R3, U = U' - W S, R4, outputs, state,
//     checkpoints, while the bulk-copy engine brings the next chunk's entry in
//     as soon as each of its buffers is free.  It is a programmatic dependent
//     of pass 1, so its launch and initial state load overlap pass 1's last
//     items.

struct Entry {                                 // byte offsets in an entry
  static constexpr uint32_t GA = 0;            // [W~; Q~] hi, lo
  static constexpr uint32_t KT = 65536;        // K^^T hi, lo, [T; M] hi, lo
  static constexpr uint32_t UP = 131072;       // U' [4 slices][64][32] fp32, the
                                               // 16-byte chunks of row t rotated by t
  static constexpr uint32_t VEC = 163840;      // e^{g_m}, e^{g_C}, e^{g_C-g_m}
  static constexpr uint32_t END = VEC + 3 * 128 * 4;
};
static_assert(Entry::END <= kTcEntryBytes && kTcEntryBytes % 1024 == 0, "entry");

struct LayP {                                  // pass 1 (two CTAs per SM)
  // [K~; Q~] hi | lo: R1's A; its K~ rows are R2's MN-major B.  128 rows, two
  // 64-channel atoms of 16 KB per split (rows 64..127 of an atom: Q~).
  static constexpr uint32_t GA_HI = 0, GA_LO = 32768;
  static constexpr uint32_t GB_HI = 65536, GB_LO = 81920;   // K^ (R1's B), 64 rows
  // E1 writes the Q~ rows and K^ to the entry from registers, so once R1 has
  // read them their space is free:
  //   V: two 64-channel atoms (TMA, MN-major) in the Q~ hi rows, 16 KB apart;
  //   the inverse's scratch, then T hi (rows 0..63 of R2's A; the A
  //   descriptor's rows 64..127 read whatever follows and land in accumulator
  //   rows nobody reads) in the Q~ lo rows of atom 0;
  //   the inverse's fp32 A and X over the Q~ lo rows of atom 1 and K^, then
  //   T lo over the start of A.
  // Before V lands, its two slots hold the images of the M rows of the
  // entry's [T; M] (hi, lo) for their bulk copy.
  static constexpr uint32_t V0 = 8192, M_HI = 8192, M_LO = 24576;
  static constexpr uint32_t PT = 40960, T_HI = 40960, T_LO = 57344;
  // Once R2 has read its operands nothing of the item is left in shared
  // memory: the next item's raw q, k, alpha rows land in [48 KB, 96 KB) (and
  // its beta box in MISC) while this item's epilogue writes the W~ and U'
  // images for their bulk copies in [0, 48 KB).  E1 reads the staged rows
  // into registers before its first barrier and writes tiles only after it.
  static constexpr uint32_t STG_Q = 49152, STG_K = 65536, STG_A = 81920;
  static constexpr uint32_t W_IMG = 0, U_IMG = 32768;  // W~ hi | lo (32 KB), U' half (16 KB)
  static constexpr uint32_t AF = 57344, XF = AF + 64 * 68 * 4;
  static constexpr uint32_t MISC = 98304;
  static constexpr uint32_t BET = MISC, GM = BET + 256, GC = GM + 512;
  static constexpr uint32_t EGC = GC + 512, ECM = EGC + 512, EGM = ECM + 512;
  static constexpr uint32_t TOT4 = EGM + 512, NSCR = TOT4 + 2048, BST = NSCR + 768;
  static constexpr uint32_t MBAR = BST + 1024, VBAR = MBAR + 8, SBAR = VBAR + 8;
  static constexpr uint32_t TSLOT = SBAR + 8, ITEM = TSLOT + 8;  // staged item: tok0, n
  static constexpr uint32_t END = ITEM + 8;
  static constexpr size_t kBytes = END + 1024;
};
static_assert(LayP::V0 % 1024 == 0 && LayP::V0 + 16384 + 8192 <= LayP::GA_LO,
              "V atoms inside the Q~ hi rows");
static_assert(LayP::PT + 3 * 1024 <= LayP::T_HI + 8192 && LayP::T_HI + 8192 <= LayP::GA_LO + 16384,
              "scratch and T hi inside the Q~ lo rows of atom 0");
static_assert(LayP::AF == LayP::GA_LO + 16384 + 8192 && LayP::XF + 64 * 68 * 4 <= LayP::MISC,
              "A and X over the Q~ lo rows of atom 1 and K^");
static_assert(LayP::T_LO + 8192 <= LayP::XF, "T lo over A only");
static_assert(LayP::STG_Q >= LayP::U_IMG + 16384 && LayP::STG_A + 16384 <= LayP::MISC &&
                  LayP::BST % 128 == 0, "staging beside the epilogue images");
static_assert(2 * (LayP::kBytes + 1024) <= 233472, "two CTAs per SM");


struct LayS {                                  // pass 2
  static constexpr uint32_t GA = 0;            // [W~; Q~] hi, lo
  // K^ (read MN-major as K^^T) hi, lo; [T; M] hi, lo
  static constexpr uint32_t KH_HI = 65536, KH_LO = 81920, TM_HI = 98304, TM_LO = 114688;
  // B operands MN-major with the hi and lo splits stacked along N (n 0..31
  // hi, 32..63 lo): one N = 64 MMA takes both products of an A split
  static constexpr uint32_t SB = 131072;       // S~: K = 128 channels x 64
  static constexpr uint32_t UT = SB + 16384;   // U: K = 64 tokens x 64
  // per chunk parity: U' slice [64][32] fp32, then the three vectors
  static constexpr uint32_t SMALL = UT + 8192, SMALL_BYTES = 8192 + 1536;
  static constexpr uint32_t MBAR = SMALL + 2 * SMALL_BYTES, G1 = MBAR + 8, G2 = G1 + 8;
  static constexpr uint32_t TSLOT = G2 + 8, END = TSLOT + 8;
  static constexpr size_t kBytes = END + 1024;
};
static_assert(LayS::SB % 1024 == 0 && LayS::UT % 1024 == 0, "pass-2 tiles");
static_assert(LayS::kBytes <= 232448, "pass-2 shared memory");

// Programmatic dependent launch: wait until the grids this one depends on
// have completed and their writes are visible (a no-op without the launch
// attribute); let the next grid on the stream start its prologue.
__device__ __forceinline__ void grid_dep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_dep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Hint: bring the box of `tm` at (x, head, tok) into L2; nothing lands in
// shared memory.
__device__ __forceinline__ void tma_prefetch3(const CUtensorMap *tm, int x, int head, int tok) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];"
               :: "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(head), "r"(tok)
               : "memory");
}

// Eight fp32 values -> one 16-byte chunk of a hi and of a lo tile image in
// global memory.
__device__ __forceinline__ void put8_global(uint8_t *hi, uint8_t *lo, const float *x) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) umma::split_bf16x2(x[2 * i], x[2 * i + 1], h[i], l[i]);
  *reinterpret_cast<uint4 *>(hi) = make_uint4(h[0], h[1], h[2], h[3]);
  *reinterpret_cast<uint4 *>(lo) = make_uint4(l[0], l[1], l[2], l[3]);
}

template <bool RAW>
__global__ void __launch_bounds__(kThreads, 2)
    prefill_tc_chunk_kernel(const PrefillParams p, const __grid_constant__ InputMaps maps) {
  extern __shared__ float4 smem4[];
  uint8_t *sm = umma::align1024(smem4);
  const uint32_t sb = umma::smem_u32(sm);
  float *bet = reinterpret_cast<float *>(sm + LayP::BET);
  float *sgm = reinterpret_cast<float *>(sm + LayP::GM);
  float *sgc = reinterpret_cast<float *>(sm + LayP::GC);
  float *tot4 = reinterpret_cast<float *>(sm + LayP::TOT4);
  float *egc = reinterpret_cast<float *>(sm + LayP::EGC);
  float *ecm = reinterpret_cast<float *>(sm + LayP::ECM);
  float *egmv = reinterpret_cast<float *>(sm + LayP::EGM);
  float *Af = reinterpret_cast<float *>(sm + LayP::AF);
  float *Xf = reinterpret_cast<float *>(sm + LayP::XF);
  uint64_t *mbar = reinterpret_cast<uint64_t *>(sm + LayP::MBAR);
  uint64_t *vbar_p = reinterpret_cast<uint64_t *>(sm + LayP::VBAR);
  uint64_t *sbar_p = reinterpret_cast<uint64_t *>(sm + LayP::SBAR);
  uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + LayP::TSLOT);

  const int tid = threadIdx.x, H = p.H;
  const int c = tid & 127, hf = tid >> 7;
  // items (chunk g, head h), g-major; this CTA takes items blockIdx.x,
  // blockIdx.x + gridDim.x, ...
  const int total = reinterpret_cast<const int *>(p.ws)[p.B] * H;
  int it = blockIdx.x;
  if (it >= total) return;
  prefetch_input_maps(maps, tid);

  if (tid < 32) umma::tmem_alloc(tslot, 256);
  if (tid == 0) {
    umma::mbar_init(mbar, 1);
    umma::mbar_init(vbar_p, 1);
    umma::mbar_init(sbar_p, 1);
  }
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tmem = *tslot;
  const uint32_t tl = tmem + ((uint32_t)(tid & 96) << 16);
  uint32_t phase = 0, vphase = 0, sphase = 0;
  // every CTA of this grid is resident from the start (two per SM, one
  // wave), so pass 2 may be scheduled now: its CTAs take SMs as this grid's
  // CTAs exit, and wait for its completion before reading the entries
  grid_dep_launch();
  const uint64_t dGA = umma::sdesc_sw128(sb);
  uint8_t *const ent0 = p.ws + prefill_tc_entries_offset(p.B);
  // TMA loads of item j's raw q, k, alpha rows and beta box into staging
  auto stage = [&](int j) {
    if (tid == 0) {
      const int gj = j / H, hj = j - (j / H) * H;
      const ChunkLoc cj = locate_chunk(p, gj, kC);
      const int tj = cj.tok0;
      // the item's rows for every thread, read after the staging barrier
      *reinterpret_cast<int2 *>(sm + LayP::ITEM) = make_int2(tj, cj.n);
      const uint32_t bar = sb + LayP::SBAR;
      mbar_expect_tx(bar, 3 * 64 * 2 * kD + 64 * 16);
      tma_load3(sb + LayP::STG_Q, &maps.q, 0, hj, tj, bar);
      tma_load3(sb + LayP::STG_K, &maps.k, 0, hj, tj, bar);
      tma_load3(sb + LayP::STG_A, &maps.a, 0, hj, tj, bar);
      tma_load2(sb + LayP::BST, &maps.b, hj & ~7, tj, bar);
    }
  };
  stage(it);
  bool ok = true, stage_owed = true, v_owed = false, mma_owed = false;  // in flight
  for (; it < total; it += gridDim.x) {
    const int g = it / H, h = it - (it / H) * H;
    uint8_t *ent = ent0 + ((size_t)g * H + h) * kTcEntryBytes;
    // every thread waits for the staged rows itself; the outcome is agreed at
    // E1's first barrier (nothing before it leaves shared memory)
    const bool gotS = own_wait(sbar_p, sphase, p.spin_limit);
    if (gotS) stage_owed = false;  // this thread's phase moved: nothing owed
    const int2 item = *reinterpret_cast<const int2 *>(sm + LayP::ITEM);
    const int t0 = item.x, n = item.y, m = n >> 1;
    if (tid == 0 && it + (int)gridDim.x < total) {  // the next item's rows into L2
      const int j = it + gridDim.x, gj = j / H, hj = j - (j / H) * H;
      const int tj = locate_chunk(p, gj, kC).tok0;
      tma_prefetch3(&maps.q, 0, hj, tj);
      tma_prefetch3(&maps.k, 0, hj, tj);
      tma_prefetch3(&maps.a, 0, hj, tj);
      tma_prefetch3(&maps.v, 0, hj, tj);
      tma_prefetch3(&maps.v, 64, hj, tj);
    }
    // ---- E1: each thread (channel pair cp, token quarter tq) reads its 16
    // tokens' q, k, alpha words from the staging area
    if (tid < kC) {
      const uint16_t bw = reinterpret_cast<const uint16_t *>(sm + LayP::BST)[tid * 8 + (h & 7)];
      const float bv = __uint_as_float((uint32_t)bw << 16);
      bet[tid] = tid < n ? (RAW ? sigmoid_f(bv) : bv) : 0.f;
    }
    const int cp = tid & 63, tq = tid >> 6, c2 = 2 * cp, tb0 = 16 * tq;
    float la0[16], la1[16];
    uint32_t kr[16], qr[16];
    {
      const uint32_t *sq = reinterpret_cast<const uint32_t *>(sm + LayP::STG_Q);
      const uint32_t *sk = reinterpret_cast<const uint32_t *>(sm + LayP::STG_K);
      const uint32_t *sa = reinterpret_cast<const uint32_t *>(sm + LayP::STG_A);
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int t = tb0 + u;
        const uint32_t aw = sa[t * 64 + cp];
        kr[u] = t < n ? sk[t * 64 + cp] : 0u;
        qr[u] = t < n ? sq[t * 64 + cp] : 0u;
        const float a0 = __uint_as_float(aw << 16), a1 = __uint_as_float(aw & 0xffff0000u);
        la0[u] = t < n ? (RAW ? neg_softplus(a0) : __logf(a0)) : 0.f;
        la1[u] = t < n ? (RAW ? neg_softplus(a1) : __logf(a1)) : 0.f;
      }
    }
    float *nscr = reinterpret_cast<float *>(sm + LayP::NSCR);   // key norms (raw inputs)
    float *nrm = nscr + 128;
    if (RAW) norm_partials(kr, nscr, tid);
#pragma unroll
    for (int u = 1; u < 16; ++u) {
      la0[u] += la0[u - 1];
      la1[u] += la1[u - 1];
    }
    tot4[tq * 128 + c2] = la0[15];
    tot4[tq * 128 + c2 + 1] = la1[15];
    if (tid == 0) umma::bulk_wait_read();  // the last item's images have been read
    // quarter sums visible; staging read (tiles writable)
    if (!(ok = __syncthreads_and(gotS) != 0)) break;
    {
      float add0 = 0.f, add1 = 0.f;
      for (int w = 0; w < tq; ++w) {
        add0 += tot4[w * 128 + c2];
        add1 += tot4[w * 128 + c2 + 1];
      }
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        la0[u] += add0;
        la1[u] += add1;
        if (tb0 + u == m) {
          sgm[c2] = la0[u];
          sgm[c2 + 1] = la1[u];
        }
      }
      if (tq == 3) {
        sgc[c2] = la0[15];
        sgc[c2 + 1] = la1[15];
      }
    }
    if (RAW) norm_finish(nscr, nrm, tid);
    __syncthreads();
    {
      const float gm0 = sgm[c2], gm1 = sgm[c2 + 1];
      if (tq == 0) {
        const float gC0 = sgc[c2], gC1 = sgc[c2 + 1];
        if (la0[0] - gm0 > 80.f || gm0 - gC0 > 80.f || la1[0] - gm1 > 80.f ||
            gm1 - gC1 > 80.f)
          set_error(p.err, KDA_DERR_RANGE);
        egc[c2] = __expf(gC0);
        egc[c2 + 1] = __expf(gC1);
        ecm[c2] = __expf(gC0 - gm0);
        ecm[c2 + 1] = __expf(gC1 - gm1);
        egmv[c2] = __expf(gm0);
        egmv[c2 + 1] = __expf(gm1);
      }
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int t = tb0 + u;
        const float f0 = __expf(la0[u] - gm0), fi0 = __expf(gm0 - la0[u]);
        const float f1 = __expf(la1[u] - gm1), fi1 = __expf(gm1 - la1[u]);
        const float kn = RAW ? nrm[t] : 1.f;
        const float k0 = __uint_as_float(kr[u] << 16) * kn;
        const float k1 = __uint_as_float(kr[u] & 0xffff0000u) * kn;
        const float q0 = __uint_as_float(qr[u] << 16);
        const float q1 = __uint_as_float(qr[u] & 0xffff0000u);
        // K~ and Q~ rows of [K~; Q~] and the K^ rows: K-major for R1, and the
        // same bytes serve R2 (K~) and the chunk walk's R4 (K^) as MN-major
        // operands, so no transposed copy is written
        uint32_t hi, lo;
        uint32_t off = umma::sw128_off16(t, c2, 128);
        umma::split_bf16x2(f0 * k0, f1 * k1, hi, lo);
        *reinterpret_cast<uint32_t *>(sm + LayP::GA_HI + off) = hi;
        *reinterpret_cast<uint32_t *>(sm + LayP::GA_LO + off) = lo;
        off = umma::sw128_off16(64 + t, c2, 128);
        umma::split_bf16x2(f0 * q0, f1 * q1, hi, lo);
        *reinterpret_cast<uint32_t *>(sm + LayP::GA_HI + off) = hi;
        *reinterpret_cast<uint32_t *>(sm + LayP::GA_LO + off) = lo;
        off = umma::sw128_off16(t, c2, 64);
        umma::split_bf16x2(fi0 * k0, fi1 * k1, hi, lo);
        *reinterpret_cast<uint32_t *>(sm + LayP::GB_HI + off) = hi;
        *reinterpret_cast<uint32_t *>(sm + LayP::GB_LO + off) = lo;
      }
    }
    tiles_ready();

    // ---- R1: G = [K~; Q~] K^^T, while the bulk-copy engine writes the Q~
    // rows (rows 64..127 of each 16 KB atom of both splits) and K^ to the
    // entry: the entry holds the tiles' shared-memory images
    if (tid == 0) {
#pragma unroll
      for (int piece = 0; piece < 4; ++piece) {
        const uint32_t off = piece * 16384 + 8192;
        umma::bulk_s2g(ent + Entry::GA + off, sb + LayP::GA_HI + off, 8192);
      }
      umma::bulk_s2g(ent + Entry::KT, sb + LayP::GB_HI, 32768);
      umma::bulk_commit();
      const uint32_t id = umma::idesc_bf16(128, 64);
      for (int ps = 0; ps < 3; ++ps) {
        const uint32_t a = ps == 1 ? LayP::GA_LO : LayP::GA_HI;
        const uint32_t b = ps == 2 ? LayP::GB_LO : LayP::GB_HI;
        for (int kk = 0; kk < 8; ++kk)
          umma::mma_bf16(tmem + kAccG, dadd(dGA, a + (kk >> 2) * 16384 + (kk & 3) * 32),
                         dadd(dGA, b + (kk >> 2) * 8192 + (kk & 3) * 32), id,
                         (uint32_t)(ps | kk));
      }
      umma::commit(mbar);
      umma::bulk_wait_read();  // before the Q~ rows and K^ are written over
    }
    mma_owed = true;
    // a barrier here, not a thread's own wait: thread 0 has waited for the
    // bulk reads of K^ and the Q~ rows, which A and the M images overwrite
    if (!(ok = tc_wait(mbar, phase, p.spin_limit))) break;
    mma_owed = false;
    {  // A = strict_tril(diag(beta) G_top) -> fp32;  M = tril(G_bottom) -> image
      float gv[32];
      umma::tmem_ld32(tl + kAccG + 32 * hf, gv);
      if (c < 64) {
        const int t = c;
        const float bt = bet[t];
#pragma unroll
        for (int s4 = 0; s4 < 8; ++s4) {
          const int s = 32 * hf + 4 * s4;
          float4 v;
          v.x = s < t ? bt * gv[4 * s4] : 0.f;
          v.y = s + 1 < t ? bt * gv[4 * s4 + 1] : 0.f;
          v.z = s + 2 < t ? bt * gv[4 * s4 + 2] : 0.f;
          v.w = s + 3 < t ? bt * gv[4 * s4 + 3] : 0.f;
          *reinterpret_cast<float4 *>(Af + fo(t, s)) = v;
        }
      } else {
        const int t = c - 64;
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          const int s = 32 * hf + 8 * ch;
          float x[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] = s + e <= t ? gv[8 * ch + e] : 0.f;
          const uint32_t off = umma::sw128_off16(t, s, 128);  // row 64 + t, less 8 KB
          put8(sm, LayP::M_HI + off, LayP::M_LO + off, x);
        }
      }
    }
    tiles_ready();
    // R1 has read the Q~ rows and K^: the M images go to the entry, then V
    // lands in their place (the Q~ hi rows) while the inverse runs
    if (tid == 0) {
      umma::bulk_s2g(ent + Entry::KT + 32768 + 8192, sb + LayP::M_HI, 8192);
      umma::bulk_s2g(ent + Entry::KT + 49152 + 8192, sb + LayP::M_LO, 8192);
      umma::bulk_commit();
      umma::bulk_wait_read();
      const uint32_t vb = sb + LayP::VBAR;
      mbar_expect_tx(vb, 2 * 64 * 128);
      tma_load3(sb + LayP::V0, &maps.v, 0, h, t0, vb);
      tma_load3(sb + LayP::V0 + 16384, &maps.v, 64, h, t0, vb);
    }
    v_owed = true;
    unit_lower_inverse(Af, Xf, reinterpret_cast<float *>(sm + LayP::PT), tid);
    {  // T = X diag(beta) -> rows 0..63 of R2's A tile and of the entry's [T; M]
      const int t = tid >> 2, s0 = (tid & 3) * 16;
      float x[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int s = s0 + e;
        x[e] = s <= t ? Xf[fo(t, s)] * bet[s] : 0.f;
      }
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const uint32_t off = umma::sw128_off16(t, s0 + 8 * hh, 128);
        put8(sm, LayP::T_HI + off, LayP::T_LO + off, x + 8 * hh);
      }
    }
    const bool gotV = own_wait(vbar_p, vphase, p.spin_limit);
    if (gotV) v_owed = false;
    if (!(ok = tiles_ready_and(gotV))) break;

    // ---- R2: T K~ -> W~ (accumulator columns 0..127);  T V -> U' (128..255).
    // K~ (rows 0..63 of [K~; Q~], 64-key atoms 16 KB apart) and V (two
    // 64-channel atoms 16 KB apart) are MN-major B operands.
    if (tid == 0) {
      // the T rows of the entry's [T; M] straight from R2's A tile
      umma::bulk_s2g(ent + Entry::KT + 32768, sb + LayP::T_HI, 8192);
      umma::bulk_s2g(ent + Entry::KT + 49152, sb + LayP::T_LO, 8192);
      umma::bulk_commit();
      const uint32_t id = umma::idesc_bf16_bmn(128, 128);
      const uint64_t dKh = umma::sdesc_sw128_mn(sb + LayP::GA_HI, 16384);
      const uint64_t dKl = umma::sdesc_sw128_mn(sb + LayP::GA_LO, 16384);
      const uint64_t dV = umma::sdesc_sw128_mn(sb + LayP::V0, 16384);
      for (int ps = 0; ps < 3; ++ps) {
        const uint32_t a = ps == 1 ? LayP::T_LO : LayP::T_HI;
        const uint64_t b = ps == 2 ? dKl : dKh;
        for (int kk = 0; kk < 4; ++kk)
          umma::mma_bf16(tmem, dadd(dGA, a + kk * 32), dadd(b, kk * 2048), id,
                         (uint32_t)(ps | kk));
      }
      for (int ps = 0; ps < 2; ++ps) {  // V is an exact bf16 input: two passes
        const uint32_t a = ps ? LayP::T_LO : LayP::T_HI;
        for (int kk = 0; kk < 4; ++kk)
          umma::mma_bf16(tmem + 128, dadd(dGA, a + kk * 32), dadd(dV, kk * 2048), id,
                         (uint32_t)(ps | kk));
      }
      umma::commit(mbar);
      umma::bulk_wait_read();  // T's images, before anything lands over them
    }
    mma_owed = true;
    // a barrier here too: thread 0 has waited for the bulk reads of T, which
    // the U' image overwrites
    if (!(ok = tc_wait(mbar, phase, p.spin_limit))) break;
    mma_owed = false;
    // R2 has read every tile: the next item's rows land during the epilogue
    if (it + (int)gridDim.x < total) {
      stage(it + gridDim.x);
      stage_owed = true;
    }
    // Epilogue: W~ (rows 0..63 of the entry's [W~; Q~]) and U' (the entry's
    // four 32-column slices, the 16-byte chunks of row t rotated by t) as
    // shared-memory images written out by the bulk-copy engine, so the
    // entry is written in whole lines: first W~ and U' slices 0, 1, then
    // slices 2, 3 in the same 16 KB once the first copies have read it.
    auto u_rows = [&](int t) {
#pragma unroll
      for (int blk = 0; blk < 4; ++blk) {
        float u[16];
        const int j0 = 64 * hf + 16 * blk;
        umma::tmem_ld16(tl + 128 + j0, u);
        float4 *row = reinterpret_cast<float4 *>(sm + LayP::U_IMG) +
                      (((j0 >> 5) - 2 * hf) * 64 + t) * 8;
#pragma unroll
        for (int e = 0; e < 4; ++e)  // chunk (j mod 32) / 4 at position (chunk + t) mod 8
          row[((((j0 & 31) >> 2) + e) + t) & 7] =
              make_float4(u[4 * e], u[4 * e + 1], u[4 * e + 2], u[4 * e + 3]);
      }
    };
    if (c < 64) {
      const int t = c;
#pragma unroll
      for (int blk = 0; blk < 4; ++blk) {
        float w[16];
        const int k0 = 64 * hf + 16 * blk;
        umma::tmem_ld16(tl + k0, w);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const uint32_t off = umma::sw128_off16(t, k0 + 8 * hh, 64);  // two 8 KB atoms
          put8(sm, LayP::W_IMG + off, LayP::W_IMG + 16384 + off, w + 8 * hh);
        }
      }
      if (hf == 0) u_rows(t);
    }
    tiles_ready();
    if (c >= 64) {
      const int j = (c - 64) + 64 * hf;  // 0..127 over the threads of lanes 64..127
      float *vec = reinterpret_cast<float *>(ent + Entry::VEC);
      vec[j] = egmv[j];
      vec[128 + j] = egc[j];
      vec[256 + j] = ecm[j];
    }
    if (tid == 0) {
#pragma unroll
      for (int piece = 0; piece < 4; ++piece)  // hi atom 0, 1, lo atom 0, 1
        umma::bulk_s2g(ent + Entry::GA + piece * 16384, sb + LayP::W_IMG + piece * 8192, 8192);
      umma::bulk_s2g(ent + Entry::UP, sb + LayP::U_IMG, 16384);
      umma::bulk_commit();
      umma::bulk_wait_read();
    }
    __syncthreads();
    if (c < 64 && hf == 1) u_rows(c);
    tiles_ready();
    if (tid == 0) {
      umma::bulk_s2g(ent + Entry::UP + 16384, sb + LayP::U_IMG, 16384);
      umma::bulk_commit();
    }
  }
  if (!ok && tid == 0) {
    set_error(p.err, KDA_DERR_TIMEOUT);
    // one more bounded chance for what is still in flight
    if ((mma_owed) && !umma::mbar_wait(mbar, phase, kDrainWaitPolls))
      set_error(p.err, KDA_DERR_UNSAFE);
    if ((v_owed) && !umma::mbar_wait(vbar_p, vphase, kDrainWaitPolls))
      set_error(p.err, KDA_DERR_UNSAFE);
    if ((stage_owed) && !umma::mbar_wait(sbar_p, sphase, kDrainWaitPolls))
      set_error(p.err, KDA_DERR_UNSAFE);
  }
  if (tid == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");  // entry writes done
  umma::fence_before_sync();
  __syncthreads();
  if (tid < 32) umma::tmem_dealloc(tmem, 256);
}

__global__ void __launch_bounds__(kThreads, 1) prefill_tc_pass_kernel(const PrefillParams p) {
  extern __shared__ float4 smem4[];
  uint8_t *sm = umma::align1024(smem4);
  const uint32_t sb = umma::smem_u32(sm);
  uint64_t *mbar = reinterpret_cast<uint64_t *>(sm + LayS::MBAR);
  uint64_t *g1bar = reinterpret_cast<uint64_t *>(sm + LayS::G1);
  uint64_t *g2bar = reinterpret_cast<uint64_t *>(sm + LayS::G2);
  uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + LayS::TSLOT);

  const int tid = threadIdx.x, sl = blockIdx.x, h = blockIdx.y, i = blockIdx.z;
  const int H = p.H, col0 = sl * kNC;
  const int c = tid & 127, hf = tid >> 7;
  // Launched as a programmatic dependent of pass 1: until grid_dep_wait()
  // returns, only what was written before pass 1 started (the chunk table,
  // the segment arrays, the pool) is read.  Every CTA waits before it exits,
  // so this grid completes after pass 1 whatever path it takes.
  const int cu0 = p.cu_seqlens[i], cu1 = p.cu_seqlens[i + 1];
  const int L = cu1 - cu0;
  const int p0 = p.start_pos ? p.start_pos[i] : 0;
  if (cu0 < 0 || L < 0 || cu1 > p.N || p0 < 0 || L == 0) {  // flagged by the table
    grid_dep_wait();
    return;
  }
  const int slot = p.state_slots[i];
  if (slot < 0 || slot >= p.P) {
    if (tid == 0 && sl == 0) set_error(p.err, KDA_DERR_SLOT);
    grid_dep_wait();
    return;
  }
  const int *table = reinterpret_cast<const int *>(p.ws);
  const int g0 = table[i], nch = table[i + 1] - table[i];
  if (nch <= 0) {
    grid_dep_wait();
    return;
  }

  if (tid < 32) umma::tmem_alloc(tslot, 128);
  if (tid == 0) {
    umma::mbar_init(mbar, 1);
    umma::mbar_init(g1bar, 1);
    umma::mbar_init(g2bar, 1);
  }
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tmem = *tslot;
  const uint32_t tl = tmem + ((uint32_t)(tid & 96) << 16);
  // TMEM columns of the R3 / R4 accumulators, 64 each: columns 0..31 take
  // the hi*hi and lo*hi products, 32..63 hi*lo and lo*lo; a result is their
  // sum
  constexpr uint32_t kA3 = 0, kA4 = 64;
  uint32_t phase = 0, ph1 = 0, ph2 = 0;
  bool owe1 = false, owe2 = false, mma_owed = false;
  const uint64_t dGA = umma::sdesc_sw128(sb);
  const uint64_t dSB = umma::sdesc_sw128_mn(sb + LayS::SB);
  const uint64_t dUT = umma::sdesc_sw128_mn(sb + LayS::UT);
  const uint8_t *ent0 = p.ws + prefill_tc_entries_offset(p.B);
  auto entry = [&](int q) { return ent0 + ((size_t)(g0 + q) * H + h) * kTcEntryBytes; };
  // buffers: [W~; Q~] and the small parts (parity q & 1); K^^T and [T; M]
  auto issue_g1 = [&](int q) {
    if (tid == 0) {
      const uint8_t *e = entry(q);
      const uint32_t bar = sb + LayS::G1, sp = sb + LayS::SMALL + (q & 1) * LayS::SMALL_BYTES;
      mbar_expect_tx(bar, 65536 + LayS::SMALL_BYTES);
      for (int k = 0; k < 4; ++k)
        umma::bulk_g2s(sb + LayS::GA + 16384 * k, e + Entry::GA + 16384 * k, 16384, bar);
      umma::bulk_g2s(sp, e + Entry::UP + sl * 8192, 8192, bar);
      umma::bulk_g2s(sp + 8192, e + Entry::VEC, 1536, bar);
    }
    owe1 = true;
  };
  auto issue_g2 = [&](int q) {
    if (tid == 0) {
      const uint8_t *e = entry(q);
      const uint32_t bar = sb + LayS::G2;
      mbar_expect_tx(bar, 65536);
      for (int k = 0; k < 4; ++k)
        umma::bulk_g2s(sb + LayS::KH_HI + 16384 * k, e + Entry::KT + 16384 * k, 16384, bar);
    }
    owe2 = true;
  };
  float S[16];
  {
    const float *src = p.pool + ((size_t)slot * H + h) * kD * kD;
#pragma unroll
    for (int jj = 0; jj < 16; ++jj)
      S[jj] = src[(size_t)(col0 + 16 * hf + jj) * kD + c];
  }
  grid_dep_wait();  // pass 1's entries are complete and visible
  issue_g1(0);
  issue_g2(0);
  const int r0 = p0 % kC;
  bool ok = true;
  for (int q = 0; q < nch; ++q) {
    const int s_loc = max(0, q * kC - r0);
    const int e_loc = min(L, (q + 1) * kC - r0);
    const int n = e_loc - s_loc, tok0 = cu0 + s_loc;
    const float *up = reinterpret_cast<const float *>(sm + LayS::SMALL +
                                                      (q & 1) * LayS::SMALL_BYTES);
    const float *vec = up + 64 * kNC;
    const bool got1 = own_wait(g1bar, ph1, p.spin_limit);  // agreed at tiles_ready_and
    if (got1) owe1 = false;  // this thread's phase moved: nothing owed
    if (tid == 32 && q + 2 < nch) {  // two chunks ahead: into L2 (not the MMA warp)
      const uint8_t *e = entry(q + 2);
      umma::prefetch_l2(e + Entry::GA, 131072);
      umma::prefetch_l2(e + Entry::UP + sl * 8192, 8192);
      umma::prefetch_l2(e + Entry::VEC, 1536);
    }
    {  // S~ = Diag(e^{g_m}) S -> S~^T tile (row j, k = channel)
      const float egm = vec[c];
      float x[16];
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) x[jj] = egm * S[jj];
      put16_mn(sm, LayS::SB, c, 16 * hf, x);
    }
    if (!(ok = tiles_ready_and(got1))) break;
    // ---- R3: [W~; Q~] S~ -> W S (rows 0..63), Q S (rows 64..127)
    if (tid == 0) {  // A_hi [S~_hi | S~_lo], then A_lo [S~_hi | S~_lo] (N = 64)
      const uint32_t id = umma::idesc_bf16_bmn(128, 2 * kNC);
      for (int ps = 0; ps < 2; ++ps) {
        const uint32_t a = ps ? LayS::GA + 32768 : LayS::GA;
        for (int kk = 0; kk < 8; ++kk)
          umma::mma_bf16(tmem + kA3, dadd(dGA, a + (kk >> 2) * 16384 + (kk & 3) * 32),
                         dadd(dSB, kk * 2048), id, (uint32_t)(ps | kk));
      }
      umma::commit(mbar);
    }
    mma_owed = true;
    // each thread sees R3 complete; the outcome is agreed at the next barrier
    // (nothing below writes global memory before it)
    const bool got3 = own_wait(mbar, phase, p.spin_limit);
    if (got3) mma_owed = false;
    if (tid == 0 && got3 && q + 1 < nch) issue_g1(q + 1);  // [W~; Q~] is free; the other parity too
    if (c < 64) {  // U = U' - W S -> U^T tile (row j, k = t)
      const int t = c;
      float ws[16];
      umma::tmem_ld16_pair_sum(tl + kA3 + 16 * hf, tl + kA3 + kNC + 16 * hf, ws);
      const float4 *u4 = reinterpret_cast<const float4 *>(up + t * kNC);
#pragma unroll
      for (int e = 0; e < 4; ++e) {  // rotated chunks: 8 rows hit 8 bank groups
        const float4 uv = u4[(4 * hf + e + t) & 7];
        ws[4 * e] = uv.x - ws[4 * e];
        ws[4 * e + 1] = uv.y - ws[4 * e + 1];
        ws[4 * e + 2] = uv.z - ws[4 * e + 2];
        ws[4 * e + 3] = uv.w - ws[4 * e + 3];
      }
      put16_mn(sm, LayS::UT, t, 16 * hf, ws);
    }
    const bool got2 = own_wait(g2bar, ph2, p.spin_limit);
    if (got2) owe2 = false;
    if (!(ok = tiles_ready_and(got2 && got3))) break;
    // ---- R4: K^^T U -> state increment; [T; M] U accumulates M U on Q S
    if (tid == 0) {  // as R3: both A splits against [U_hi | U_lo]; K^^T is the
                     // K^ tile read MN-major (64-key atoms 8 KB apart)
      const uint32_t idk = umma::idesc_bf16_abmn(128, 2 * kNC);
      const uint32_t id = umma::idesc_bf16_bmn(128, 2 * kNC);
      for (int ps = 0; ps < 2; ++ps) {
        const uint64_t a = umma::sdesc_sw128_mn(sb + (ps ? LayS::KH_LO : LayS::KH_HI), 8192);
        for (int kk = 0; kk < 4; ++kk)
          umma::mma_bf16(tmem + kA4, dadd(a, kk * 2048), dadd(dUT, kk * 2048), idk,
                         (uint32_t)(ps | kk));
      }
      for (int ps = 0; ps < 2; ++ps) {
        const uint32_t a = ps ? LayS::TM_LO : LayS::TM_HI;
        for (int kk = 0; kk < 4; ++kk)
          umma::mma_bf16(tmem + kA3, dadd(dGA, a + kk * 32), dadd(dUT, kk * 2048), id, 1u);
      }
      umma::commit(mbar);
    }
    mma_owed = true;
    if (!(ok = tc_wait(mbar, phase, p.spin_limit))) break;
    mma_owed = false;
    if (q + 1 < nch) issue_g2(q + 1);  // K^ and [T; M] are free
    {
      // the increment's two halves, and (warps of rows 64..127) the outputs'
      // two halves, loaded together with one wait
      float acc[16], o[16];
      if (c >= 64)
        umma::tmem_ld16_pair_sum2(tl + kA4 + 16 * hf, tl + kA4 + kNC + 16 * hf,
                                  tl + kA3 + 16 * hf, tl + kA3 + kNC + 16 * hf, acc, o);
      else
        umma::tmem_ld16_pair_sum(tl + kA4 + 16 * hf, tl + kA4 + kNC + 16 * hf, acc);
      const float a1 = vec[128 + c], a2 = vec[256 + c];
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) S[jj] = fmaf(a1, S[jj], a2 * acc[jj]);
      if (c >= 64) {  // outputs of row t = c - 64
        const int t = c - 64;
        if (t < n) {
          float4 *dst = reinterpret_cast<float4 *>(
              p.o + ((size_t)(tok0 + t) * H + h) * kD + col0 + 16 * hf);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            dst[e] = make_float4(o[4 * e], o[4 * e + 1], o[4 * e + 2], o[4 * e + 3]);
        }
      }
    }
    const int P_end = p0 + e_loc;
    if (p.ckpt_every > 0 && P_end % p.ckpt_every == 0 && p.ckpt_slots) {
      const int mth = P_end / p.ckpt_every - p0 / p.ckpt_every - 1;
      if (mth >= 0 && mth < p.max_ckpt) {
        const int cs = p.ckpt_slots[(size_t)i * p.max_ckpt + mth];
        if (cs >= p.P) {
          if (tid == 0 && sl == 0) set_error(p.err, KDA_DERR_SLOT);
        } else if (cs >= 0) {
          float *dst = p.pool + ((size_t)cs * H + h) * kD * kD;
#pragma unroll
          for (int jj = 0; jj < 16; ++jj)
            dst[(size_t)(col0 + 16 * hf + jj) * kD + c] = S[jj];
        }
      }
    }
    // no barrier here: the next chunk's tiles_ready_and() orders this
    // chunk's TMEM reads before the next MMAs
  }
  if (!ok) {
    if (tid == 0) {
      set_error(p.err, KDA_DERR_TIMEOUT);
      if ((mma_owed) && !umma::mbar_wait(mbar, phase, kDrainWaitPolls))
        set_error(p.err, KDA_DERR_UNSAFE);
    }
  } else {
    float *dst = p.pool + ((size_t)slot * H + h) * kD * kD;
#pragma unroll
    for (int jj = 0; jj < 16; ++jj) dst[(size_t)(col0 + 16 * hf + jj) * kD + c] = S[jj];
  }
  // no copy into shared memory outlives the CTA
  if (tid == 0) {
    if ((owe1) && !umma::mbar_wait(g1bar, ph1, kDrainWaitPolls))
      set_error(p.err, KDA_DERR_UNSAFE);
    if ((owe2) && !umma::mbar_wait(g2bar, ph2, kDrainWaitPolls))
      set_error(p.err, KDA_DERR_UNSAFE);
  }
  umma::fence_before_sync();
  __syncthreads();
  if (tid < 32) umma::tmem_dealloc(tmem, 128);
}
}  // namespace

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t,
                                  void *, const cuuint64_t *, const cuuint64_t *,
                                  const cuuint32_t *, const cuuint32_t *,
                                  CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled from the driver, looked up once.
EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// [N][H][D] bf16 as a 3-D tensor map with boxes of `box_x` channels x 1 head
// x 64 tokens, zero fill past N; no swizzle, or (box_x = 64) the 128-byte
// swizzle of an MN-major MMA operand (one 64-channel atom per box).
cudaError_t input_map(CUtensorMap *tm, const void *base, int N, int H, int box_x,
                      bool swizzle128 = false) {
  EncodeTiledFn enc = encode_tiled();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t gdim[3] = {(cuuint64_t)kD, (cuuint64_t)H, (cuuint64_t)N};
  const cuuint64_t gstride[2] = {(cuuint64_t)kD * 2, (cuuint64_t)H * kD * 2};
  const cuuint32_t box[3] = {(cuuint32_t)box_x, 1, (cuuint32_t)kC};
  const cuuint32_t estride[3] = {1, 1, 1};
  const CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base),
                         gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// beta [N][H] bf16 as a 2-D tensor map with boxes of 8 heads x 64 tokens
// (H a multiple of 8: the row stride must be a multiple of 16 bytes).
cudaError_t beta_map(CUtensorMap *tm, const void *base, int N, int H) {
  EncodeTiledFn enc = encode_tiled();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t gdim[2] = {(cuuint64_t)H, (cuuint64_t)N};
  const cuuint64_t gstride[1] = {(cuuint64_t)H * 2};
  const cuuint32_t box[2] = {8, (cuuint32_t)kC};
  const cuuint32_t estride[2] = {1, 1};
  const CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base),
                         gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

// d_k = d_v = 128, chunk 64, bf16 inputs, H a multiple of 8: two passes
// through the workspace when one is given, else the fused single pass.
cudaError_t launch_prefill_tc(const PrefillParams &p, cudaStream_t s) {
  if (p.B == 0 || p.N == 0) return cudaSuccess;
  const bool two = p.ws != nullptr;
  InputMaps maps;
  cudaError_t e = input_map(&maps.q, p.q, p.N, p.H, kD);
  if (e == cudaSuccess) e = input_map(&maps.k, p.k, p.N, p.H, kD);
  if (e == cudaSuccess) e = input_map(&maps.a, p.alpha, p.N, p.H, kD);
  if (e == cudaSuccess)
    e = two ? input_map(&maps.v, p.v, p.N, p.H, 64, true) : input_map(&maps.v, p.v, p.N, p.H, kNC);
  if (e == cudaSuccess) e = beta_map(&maps.b, p.beta, p.N, p.H);
  if (e != cudaSuccess) return e;
  if (!two) {
    auto k1 = p.raw ? prefill_tc_kernel<true> : prefill_tc_kernel<false>;
    e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Lay::kBytes);
    if (e != cudaSuccess) return e;
    k1<<<dim3(kD / kNC, p.H, p.B), kThreads, Lay::kBytes, s>>>(p, maps);
    return cudaGetLastError();
  }
  e = launch_chunk_table(p, kC, s);
  if (e != cudaSuccess) return e;
  auto kp1 = p.raw ? prefill_tc_chunk_kernel<true> : prefill_tc_chunk_kernel<false>;
  e = cudaFuncSetAttribute(kp1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)LayP::kBytes);
  // all of the unified L1 / shared-memory array as shared memory: room for
  // two CTAs per SM
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kp1, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(prefill_tc_pass_kernel,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)LayS::kBytes);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  // two CTAs per SM walk the (chunk, head) items (the last ones exit at once)
  const long long items = (long long)p.max_chunks * p.H;
  const int grid1 = (int)(items < 2LL * sms ? items : 2LL * sms);
  kp1<<<grid1, kThreads, LayP::kBytes, s>>>(p, maps);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // pass 2 as a programmatic dependent of pass 1 (its prologue overlaps
  // pass 1's last items)
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kD / kNC, p.H, p.B);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = LayS::kBytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, prefill_tc_pass_kernel, p);
}

}  // namespace kda
