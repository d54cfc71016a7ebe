// Chunked prefill on the tensor cores (tcgen05, accumulators in TMEM) for
// d_k = d_v = 128, chunk 64, bf16 inputs, with the in-pass checkpoints of
// "KDA checkpoints stay inside the prefill" (vLLM Kimi K3 optimisation page).
//
// One CTA per (value-column slice of NC columns, head, sequence) walks the
// sequence's chunks in order; nothing goes through a workspace.  Per chunk of
// C tokens with g_t = sum_{s<=t} log alpha_s (per key channel) and a
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
// Precision: every operand that is not an exact bf16 input is split into
// bf16 hi + lo and each product runs as hi*hi + lo*hi + hi*lo (three
// kind::f16 MMAs into one fp32 accumulator, ~2^-16 relative per product); V
// is an exact bf16 input and takes two.  The state stays fp32 in registers.
//
// Shared-memory operand tiles are K-major with the 128-byte swizzle (see
// kda_umma.cuh); the TMEM accumulators sit at fixed columns.
#include "kda_internal.cuh"
#include "kda_umma.cuh"

namespace kda {

namespace {

constexpr int kD = 128, kC = 64, kNC = 32, kThreads = 256;
constexpr int kSpin = 1 << 22;  // polls of a tensor-core completion barrier

// Byte offsets from a 1024-byte aligned base.
struct Lay {
  static constexpr uint32_t GA_HI = 0;       // [K~; Q~] then [W~; Q~]: 128 x 128
  static constexpr uint32_t GA_LO = 32768;
  static constexpr uint32_t GB_HI = 65536;   // K^: 64 x 128
  static constexpr uint32_t GB_LO = 81920;
  static constexpr uint32_t AF = 65536;      // after R1: A fp32 64 x 64
  static constexpr uint32_t XF = 81920;      //           X fp32 64 x 64
  static constexpr uint32_t UT_HI = 65536;   // after the solve: U^T NC x 64
  static constexpr uint32_t UT_LO = UT_HI + kNC * 128;
  static constexpr uint32_t B2_HI = 98304;   // [K~^T; V^T]: (128 + NC) x 64
  static constexpr uint32_t B2_LO = B2_HI + (128 + kNC) * 128;  // K~^T lo
  static constexpr uint32_t KH_HI = B2_LO + 16384;  // K^^T: 128 x 64
  static constexpr uint32_t KH_LO = KH_HI + 16384;
  static constexpr uint32_t TM_HI = KH_LO + 16384;  // [T; M]: 128 x 64
  static constexpr uint32_t TM_LO = TM_HI + 16384;
  static constexpr uint32_t SB_HI = TM_LO + 16384;  // S~^T: NC x 128
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
  static constexpr uint32_t MBAR = TOT4 + 2048;      // u64
  static constexpr uint32_t TSLOT = MBAR + 8;        // u32
  static constexpr uint32_t END = TSLOT + 8;
  static constexpr size_t kBytes = END + 1024;       // + alignment slack
};
static_assert(Lay::B2_LO % 1024 == 0 && Lay::KH_HI % 1024 == 0 &&
                  Lay::SB_HI % 1024 == 0 && Lay::UT_LO % 1024 == 0,
              "tiles on 1024-byte boundaries");
static_assert(Lay::UT_LO + kNC * 128 <= Lay::B2_HI, "U^T fits the K^ region");
// The next chunk's raw rows are staged while this chunk's R3/R4 run, in
// regions free from the end of R2 to the next E1: q, k (bf16 [64][128]) in
// the R2 B tile, alpha in the X array, the V slice after U^T.
constexpr uint32_t kStgQ = Lay::B2_HI, kStgK = Lay::B2_HI + 16384;
constexpr uint32_t kStgA = Lay::XF, kStgV = Lay::UT_LO + kNC * 128;
static_assert(kStgK + 16384 <= Lay::B2_HI + (128 + kNC) * 128 + 16384, "q, k staging");
static_assert(kStgV + 64 * kNC * 2 <= Lay::XF, "V staging");
static_assert(Lay::kBytes <= 232448, "shared memory per CTA");

// TMEM columns of the accumulators (512 allocated).
constexpr uint32_t kAccG = 0, kAcc2 = 64, kAcc3 = 64 + 128 + kNC,
                   kAcc4 = kAcc3 + kNC;
static_assert(kAcc4 + kNC <= 512, "TMEM columns");

// Swizzled index of element (r, c) of a 64 x 64 fp32 array (16-byte chunks
// permuted by row so that row-parallel float4 accesses avoid bank conflicts).
__device__ __forceinline__ int fo(int r, int c) {
  return r * 64 + ((((c >> 2) ^ (r & 7)) << 2) | (c & 3));
}

__device__ __forceinline__ void st_u16(uint8_t *base, uint32_t off, uint16_t v) {
  *reinterpret_cast<uint16_t *>(base + off) = v;
}
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

// Four consecutive entries (r, c..c+3) of a swizzled 64 x 64 fp32 array
// (c a multiple of 4).
__device__ __forceinline__ float4 ld4(const float *M, int r, int c) {
  return *reinterpret_cast<const float4 *>(M + fo(r, c));
}

// One block distance d of the off-diagonal pass: for the 4 - d blocks
// (a, b) = (blk + d, blk), P_ab = sum_{b<=r<a} A_ar X_rb (16 x 16 each, one
// element per thread and loop trip; operands loaded before the FMAs).
template <int d>
__device__ __forceinline__ void offdiag_sum(const float *A, const float *X,
                                            float *P, int tid) {
#pragma unroll
  for (int it = 0; it < (4 - d) * 256 / kThreads; ++it) {
    const int e = tid + it * kThreads;
    if (e < (4 - d) * 256) {
      const int blk = e >> 8, i = (e >> 4) & 15, j = e & 15;
      const int a = blk + d, b = blk;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int rr = 0; rr < d; ++rr) {
        const int rb = b + rr;
        float4 av[4];
        float xv[16];
#pragma unroll
        for (int k = 0; k < 4; ++k) av[k] = ld4(A, 16 * a + i, 16 * rb + 4 * k);
#pragma unroll
        for (int r = 0; r < 16; ++r) xv[r] = X[fo(16 * rb + r, 16 * b + j)];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          acc[0] = fmaf(av[k].x, xv[4 * k], acc[0]);
          acc[1] = fmaf(av[k].y, xv[4 * k + 1], acc[1]);
          acc[2] = fmaf(av[k].z, xv[4 * k + 2], acc[2]);
          acc[3] = fmaf(av[k].w, xv[4 * k + 3], acc[3]);
        }
      }
      P[blk * 256 + i * 16 + j] = (acc[0] + acc[1]) + (acc[2] + acc[3]);
    }
  }
}

// X_ab = -X_aa P_ab for the blocks of distance d.
template <int d>
__device__ __forceinline__ void offdiag_apply(const float *P, float *X, int tid) {
#pragma unroll
  for (int it = 0; it < (4 - d) * 256 / kThreads; ++it) {
    const int e = tid + it * kThreads;
    if (e < (4 - d) * 256) {
      const int blk = e >> 8, i = (e >> 4) & 15, j = e & 15;
      const int a = blk + d, b = blk;
      float4 xv[4];
      float pv[16];
#pragma unroll
      for (int k = 0; k < 4; ++k) xv[k] = ld4(X, 16 * a + i, 16 * a + 4 * k);
#pragma unroll
      for (int r = 0; r < 16; ++r) pv[r] = P[blk * 256 + r * 16 + j];
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        acc[0] = fmaf(xv[k].x, pv[4 * k], acc[0]);
        acc[1] = fmaf(xv[k].y, pv[4 * k + 1], acc[1]);
        acc[2] = fmaf(xv[k].z, pv[4 * k + 2], acc[2]);
        acc[3] = fmaf(xv[k].w, pv[4 * k + 3], acc[3]);
      }
      X[fo(16 * a + i, 16 * b + j)] = -((acc[0] + acc[1]) + (acc[2] + acc[3]));
    }
  }
}

// X = (I + A)^{-1} for a strictly lower-triangular 64 x 64 A (swizzled fp32
// arrays), by 16 x 16 blocks: diagonal blocks by forward substitution (one
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

__device__ __forceinline__ uint64_t dsc(uint32_t addr) {
  return umma::sdesc_sw128(addr);
}

// Thread 0 waits for the last commit (bounded); every thread learns whether
// it completed.  On success the phase advances.
__device__ __forceinline__ bool tc_wait(uint64_t *mbar, uint32_t &phase, int tid) {
  const bool ok = tid == 0 ? umma::mbar_wait(mbar, phase, kSpin) : true;
  const bool all = __syncthreads_and(ok) != 0;
  if (all) phase ^= 1u;
  umma::fence_after_sync();
  return all;
}

// Publish this thread's shared-memory tile writes to the tensor core and
// meet the MMA-issuing thread.
__device__ __forceinline__ void tiles_ready() {
  umma::fence_smem_to_async();
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
}

// 16-byte global -> shared copy; src_bytes = 0 writes zeros (src unread).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src,
                                           int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;"
               :: "r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;"
               :: "l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ float bf(const __nv_bfloat16 *p) {
  return __bfloat162float(*p);
}

__global__ void __launch_bounds__(kThreads, 1) prefill_tc_kernel(const PrefillParams p) {
  extern __shared__ float4 smem4[];
  uint8_t *sm = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem4) + 1023) & ~(uintptr_t)1023);
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
  if (tid == 0) umma::mbar_init(mbar, 1);
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tmem = *tslot;
  const uint32_t tl = tmem + ((uint32_t)(tid & 96) << 16);  // lane quadrant
  uint32_t phase = 0;

  // S[c][col0 + 16 hf + jj], fp32, for the whole pass
  float S[16];
  {
    const float *src = p.pool + ((size_t)slot * H + h) * kD * kD;
#pragma unroll
    for (int jj = 0; jj < 16; ++jj)
      S[jj] = src[(size_t)(col0 + 16 * hf + jj) * kD + c];
  }
  const __nv_bfloat16 *qin = reinterpret_cast<const __nv_bfloat16 *>(p.q);
  const __nv_bfloat16 *kin = reinterpret_cast<const __nv_bfloat16 *>(p.k);
  const __nv_bfloat16 *vin = reinterpret_cast<const __nv_bfloat16 *>(p.v);
  const __nv_bfloat16 *ain = reinterpret_cast<const __nv_bfloat16 *>(p.alpha);
  const __nv_bfloat16 *bin = reinterpret_cast<const __nv_bfloat16 *>(p.beta);

  const int r0 = p0 % kC;
  const int nch = (r0 + L + kC - 1) / kC;
  // Copies of chunk qq's raw rows into the staging areas (rows past the
  // chunk read as zeros), its beta into a register, and an L2 prefetch of
  // chunk qq + 1's rows.
  float beta_next = 0.f;
  auto stage = [&](int qq) {
    const int s0 = max(0, qq * kC - r0), nn = min(L, (qq + 1) * kC - r0) - s0;
    const size_t row0 = ((size_t)(cu0 + s0) * H + h) * kD;
    for (int e = tid; e < 3 * 64 * 16; e += kThreads) {
      const int tens = e >> 10, t = (e >> 4) & 63, ch = e & 15;
      const __nv_bfloat16 *src = (tens == 0 ? qin : tens == 1 ? kin : ain) + row0 +
                                 (size_t)min(t, nn - 1) * H * kD + ch * 8;
      cp_async16(sb + (tens == 0 ? kStgQ : tens == 1 ? kStgK : kStgA) + t * 256 + ch * 16,
                 src, t < nn ? 16 : 0);
    }
    {
      const int t = tid >> 2, ch = tid & 3;
      cp_async16(sb + kStgV + t * 64 + ch * 16,
                 vin + row0 + (size_t)min(t, nn - 1) * H * kD + col0 + ch * 8,
                 t < nn ? 16 : 0);
    }
    cp_async_commit();
    if (tid < kC)
      beta_next = tid < nn ? bf(bin + (size_t)(cu0 + s0 + tid) * H + h) : 0.f;
    if (qq + 1 < nch) {
      const int s1 = (qq + 1) * kC - r0, e1 = min(L, s1 + kC);
      const int t = tid & 63, tens = tid >> 6;
      if (s1 + t < e1) {
        const size_t r = ((size_t)(cu0 + s1 + t) * H + h) * kD;
        if (tens < 3)
          prefetch_l2((tens == 0 ? qin : tens == 1 ? kin : ain) + r, 256);
        else
          prefetch_l2(vin + r + col0, 2 * kNC);
      }
    }
  };
  stage(0);
  bool ok = true;
  for (int q = 0; q < nch; ++q) {
    const int s_loc = max(0, q * kC - r0);
    const int e_loc = min(L, (q + 1) * kC - r0);
    const int n = e_loc - s_loc, tok0 = cu0 + s_loc, m = n >> 1;

    // ---- E1: the chunk's raw rows are in the staging areas.  Thread
    // (channel pair cp, token quarter tq) takes channels 2cp, 2cp+1 of rows
    // 16tq .. 16tq+15: cumulative log-decay (padded rows: alpha = 1), then the
    // scaled operand tiles; S~ from the state rows this thread owns.
    cp_async_wait_all();
    if (tid < kC) bet[tid] = beta_next;
    __syncthreads();
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
        kr[u] = sk[t * 64 + cp];
        qr[u] = sq[t * 64 + cp];
        la0[u] = t < n ? __logf(__uint_as_float(aw << 16)) : 0.f;
        la1[u] = t < n ? __logf(__uint_as_float(aw & 0xffff0000u)) : 0.f;
      }
    }
    uint32_t vw[4];
    {
      const int j = tid & 31, tg = tid >> 5;
      const uint16_t *vs = reinterpret_cast<const uint16_t *>(sm + kStgV);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int ta = 8 * tg + 2 * e;
        vw[e] = (uint32_t)vs[ta * kNC + j] | ((uint32_t)vs[(ta + 1) * kNC + j] << 16);
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
      float kt0[8], kt1[8], kh0[8], kh1[8];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int t = tb0 + u;
        const float f0 = __expf(la0[u] - gm0), fi0 = __expf(gm0 - la0[u]);
        const float f1 = __expf(la1[u] - gm1), fi1 = __expf(gm1 - la1[u]);
        const float k0 = __uint_as_float(kr[u] << 16);
        const float k1 = __uint_as_float(kr[u] & 0xffff0000u);
        const float q0 = __uint_as_float(qr[u] << 16);
        const float q1 = __uint_as_float(qr[u] & 0xffff0000u);
        uint32_t hi, lo;
        uint32_t off = umma::sw128_off16(t, c2, 128);
        umma::split_bf16x2(f0 * k0, f1 * k1, hi, lo);
        *reinterpret_cast<uint32_t *>(sm + Lay::GA_HI + off) = hi;
        *reinterpret_cast<uint32_t *>(sm + Lay::GA_LO + off) = lo;
        off = umma::sw128_off16(64 + t, c2, 128);
        umma::split_bf16x2(f0 * q0, f1 * q1, hi, lo);
        *reinterpret_cast<uint32_t *>(sm + Lay::GA_HI + off) = hi;
        *reinterpret_cast<uint32_t *>(sm + Lay::GA_LO + off) = lo;
        off = umma::sw128_off16(t, c2, 64);
        umma::split_bf16x2(fi0 * k0, fi1 * k1, hi, lo);
        *reinterpret_cast<uint32_t *>(sm + Lay::GB_HI + off) = hi;
        *reinterpret_cast<uint32_t *>(sm + Lay::GB_LO + off) = lo;
        kt0[u & 7] = f0 * k0;
        kt1[u & 7] = f1 * k1;
        kh0[u & 7] = fi0 * k0;
        kh1[u & 7] = fi1 * k1;
        if ((u & 7) == 7) {
          const int tb = t - 7;
          put8(sm, Lay::B2_HI + umma::sw128_off16(c2, tb, 128 + kNC),
               Lay::B2_LO + umma::sw128_off16(c2, tb, 128), kt0);
          put8(sm, Lay::B2_HI + umma::sw128_off16(c2 + 1, tb, 128 + kNC),
               Lay::B2_LO + umma::sw128_off16(c2 + 1, tb, 128), kt1);
          put8(sm, Lay::KH_HI + umma::sw128_off16(c2, tb, 128),
               Lay::KH_LO + umma::sw128_off16(c2, tb, 128), kh0);
          put8(sm, Lay::KH_HI + umma::sw128_off16(c2 + 1, tb, 128),
               Lay::KH_LO + umma::sw128_off16(c2 + 1, tb, 128), kh1);
        }
      }
    }
    {
      const float egm = __expf(sgm[c]);
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) {
        uint16_t hi, lo;
        umma::split_bf16(egm * S[jj], hi, lo);
        const uint32_t off = umma::sw128_off16(16 * hf + jj, c, kNC);
        st_u16(sm, Lay::SB_HI + off, hi);
        st_u16(sm, Lay::SB_LO + off, lo);
      }
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
        const uint32_t a = sb + (ps == 1 ? Lay::GA_LO : Lay::GA_HI);
        const uint32_t b = sb + (ps == 2 ? Lay::GB_LO : Lay::GB_HI);
        for (int kk = 0; kk < 8; ++kk)
          umma::mma_bf16(tmem + kAccG, dsc(a + (kk >> 2) * 16384 + (kk & 3) * 32),
                         dsc(b + (kk >> 2) * 8192 + (kk & 3) * 32), id,
                         (uint32_t)(ps | kk));
      }
      umma::commit(mbar);
    }
    if (!(ok = tc_wait(mbar, phase, tid))) break;
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
        const uint32_t a = sb + (ps == 1 ? Lay::TM_LO : Lay::TM_HI);
        const uint32_t b = sb + (ps == 2 ? Lay::B2_LO : Lay::B2_HI);
        const uint32_t id = umma::idesc_bf16(128, ps == 2 ? 128 : 128 + kNC);
        for (int kk = 0; kk < 4; ++kk)
          umma::mma_bf16(tmem + kAcc2, dsc(a + kk * 32), dsc(b + kk * 32), id,
                         (uint32_t)(ps | kk));
      }
      umma::commit(mbar);
    }
    if (!(ok = tc_wait(mbar, phase, tid))) break;
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
    if (tid == 0) {
      const uint32_t id = umma::idesc_bf16(128, kNC);
      for (int ps = 0; ps < 3; ++ps) {
        const uint32_t a = sb + (ps == 1 ? Lay::GA_LO : Lay::GA_HI);
        const uint32_t b = sb + (ps == 2 ? Lay::SB_LO : Lay::SB_HI);
        for (int kk = 0; kk < 8; ++kk)
          umma::mma_bf16(tmem + kAcc3, dsc(a + (kk >> 2) * 16384 + (kk & 3) * 32),
                         dsc(b + (kk >> 2) * (kNC * 128) + (kk & 3) * 32), id,
                         (uint32_t)(ps | kk));
      }
      umma::commit(mbar);
    }
    if (!(ok = tc_wait(mbar, phase, tid))) break;
    if (c < 64) {  // U = U' - W S -> U^T tile (row j, k = t)
      const int t = c;
      float ws[16];
      umma::tmem_ld16(tl + kAcc3 + 16 * hf, ws);
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) {
        uint16_t hi, lo;
        umma::split_bf16(up[jj] - ws[jj], hi, lo);
        const uint32_t off = umma::sw128_off16(16 * hf + jj, t, kNC);
        st_u16(sm, Lay::UT_HI + off, hi);
        st_u16(sm, Lay::UT_LO + off, lo);
      }
    }
    tiles_ready();

    // ---- R4: K^^T U -> state increment; [T; M] U accumulates M U on Q S
    if (tid == 0) {
      const uint32_t id = umma::idesc_bf16(128, kNC);
      for (int ps = 0; ps < 3; ++ps) {
        const uint32_t a = sb + (ps == 1 ? Lay::KH_LO : Lay::KH_HI);
        const uint32_t b = sb + (ps == 2 ? Lay::UT_LO : Lay::UT_HI);
        for (int kk = 0; kk < 4; ++kk)
          umma::mma_bf16(tmem + kAcc4, dsc(a + kk * 32), dsc(b + kk * 32), id,
                         (uint32_t)(ps | kk));
      }
      for (int ps = 0; ps < 3; ++ps) {
        const uint32_t a = sb + (ps == 1 ? Lay::TM_LO : Lay::TM_HI);
        const uint32_t b = sb + (ps == 2 ? Lay::UT_LO : Lay::UT_HI);
        for (int kk = 0; kk < 4; ++kk)
          umma::mma_bf16(tmem + kAcc3, dsc(a + kk * 32), dsc(b + kk * 32), id, 1u);
      }
      umma::commit(mbar);
    }
    if (!(ok = tc_wait(mbar, phase, tid))) break;
    {
      float acc[16];
      umma::tmem_ld16(tl + kAcc4 + 16 * hf, acc);
      const float a1 = egc[c], a2 = ecm[c];
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) S[jj] = fmaf(a1, S[jj], a2 * acc[jj]);
      if (c >= 64) {  // outputs of row t = c - 64
        float o[16];
        umma::tmem_ld16(tl + kAcc3 + 16 * hf, o);
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
      umma::mbar_wait(mbar, phase, 1 << 26);
    }
  } else {
    float *dst = p.pool + ((size_t)slot * H + h) * kD * kD;
#pragma unroll
    for (int jj = 0; jj < 16; ++jj) dst[(size_t)(col0 + 16 * hf + jj) * kD + c] = S[jj];
  }
  cp_async_wait_all();  // no copy into shared memory outlives the CTA
  umma::fence_before_sync();
  __syncthreads();
  if (tid < 32) umma::tmem_dealloc(tmem, 512);
}

}  // namespace

// d_k = d_v = 128, chunk 64, bf16 inputs; no workspace.
cudaError_t launch_prefill_tc(const PrefillParams &p, cudaStream_t s) {
  if (p.B == 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)Lay::kBytes);
  if (e != cudaSuccess) return e;
  prefill_tc_kernel<<<dim3(kD / kNC, p.H, p.B), kThreads, Lay::kBytes, s>>>(p);
  return cudaGetLastError();
}

}  // namespace kda
