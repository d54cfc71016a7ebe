// The single-token step of the recurrence on a register-resident state
// slice, shared by every kernel that advances a committed state (replay,
// ordinary decode, materialize, the direct-snapshot ablation), so identical
// inputs give identical bits whichever kernel runs them.
//
// Thread mapping (head dim D = d_k = d_v): thread t of a group of 2*D threads
// owns value columns j0 = 2*(t/4), j0+1 and, of each, key rows
// c = 4*(rg + 4*i) + e, rg = t % 4, i < D/16, e < 4.  Rows are held as pairs
// (c, c+1) in 64-bit registers and advanced with packed fp32x2 instructions;
// the four threads of a column reduce with two xor-shuffles in a fixed order.
#pragma once

#include "kda_internal.cuh"

namespace kda {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kTMax = 16;  // longest speculative segment (ring depth limit)

typedef unsigned long long f2;  // two fp32 lanes

__device__ __forceinline__ f2 fma2(f2 a, f2 b, f2 c) {
  f2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ f2 mul2(f2 a, f2 b) {
  f2 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f2 pack2(float x, float y) {
  f2 d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(x), "f"(y));
  return d;
}
__device__ __forceinline__ float sum2(f2 a) {  // lane0 + lane1, round to nearest
  float x, y;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(x), "=f"(y) : "l"(a));
  return __fadd_rn(x, y);
}

// Per-token record in shared memory, in the input dtype (the values exactly
// as they were given): k[D] alpha[D] q[D] v[D] beta, padded to 16 bytes.
template <int D, typename Tin>
struct Rec {
  static constexpr int kStride = 4 * D + 16 / (int)sizeof(Tin);
  static constexpr int kK = 0, kA = D, kQ = 2 * D, kV = 3 * D, kB = 4 * D;
  static constexpr int kBytes = kStride * (int)sizeof(Tin);
};

// Channels c .. c+3 of a record vector (c a multiple of 4) as two fp32 pairs
// (c, c+1) and (c+2, c+3); exact for both input dtypes.
__device__ __forceinline__ void ld4x(const float *p, f2 &a, f2 &b) {
  const ulonglong2 v = *reinterpret_cast<const ulonglong2 *>(p);
  a = v.x;
  b = v.y;
}
__device__ __forceinline__ void ld4x(const __nv_bfloat16 *p, f2 &a, f2 &b) {
  const uint2 v = *reinterpret_cast<const uint2 *>(p);
  a = pack2(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u));
  b = pack2(__uint_as_float(v.y << 16), __uint_as_float(v.y & 0xffff0000u));
}
// The same four channels as a float4.
__device__ __forceinline__ float4 ld4f(const float *p) {
  return *reinterpret_cast<const float4 *>(p);
}
__device__ __forceinline__ float4 ld4f(const __nv_bfloat16 *p) {
  const uint2 v = *reinterpret_cast<const uint2 *>(p);
  return make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u),
                     __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xffff0000u));
}

// One token of the recurrence on the thread's slice of S, fixed rounding:
//   S' = Diag(alpha) S;  dot_j = sum_c k_c S'_cj;  delta_j = beta (v_j - dot_j)
//   S  = S' + k delta^T;  o_j = sum_c q_c S_cj  (when WANT_O)
// The token's vectors are given by pointer (k, alpha, q, v and beta, in the
// input dtype, shared memory).  The only code that advances a committed
// state: replay, decode and materialize all call it, so identical inputs
// give identical bits.
// (k, alpha and q may be held in fp32 while v and beta stay in the input
// dtype: every conversion to fp32 is exact, so the bits do not change.)
// HOIST loads the step's k and alpha for all of the thread's rows before the
// arithmetic (32 more registers, one load latency per step instead of one per
// row group); the arithmetic and its order are the same either way.
template <int D, bool WANT_O, typename Tin, typename TinV = Tin, bool HOIST = false>
__device__ __forceinline__ void kda_step_ptrs(f2 (&S)[2][D / 8], const Tin *kp,
                                              const Tin *ap, const Tin *qp,
                                              const TinV *vp, const TinV *bp, int rg,
                                              int j0, float &o0, float &o1) {
  constexpr int F = D / 16;
  constexpr int NH = HOIST ? F : 1;
  f2 kh[2 * NH], ah[2 * NH];
  if (HOIST) {
#pragma unroll
    for (int f = 0; f < NH; ++f) {
      ld4x(kp + 4 * (rg + 4 * f), kh[2 * f], kh[2 * f + 1]);
      ld4x(ap + 4 * (rg + 4 * f), ah[2 * f], ah[2 * f + 1]);
    }
  }
  const float beta = in_scalar<TinV>(bp);
  const float v0 = in_scalar<TinV>(vp + j0), v1 = in_scalar<TinV>(vp + j0 + 1);
  f2 dA0 = 0, dB0 = 0, dA1 = 0, dB1 = 0;
#pragma unroll
  for (int f = 0; f < F; ++f) {
    ulonglong2 kk, aa;
    if (HOIST) {
      kk = make_ulonglong2(kh[2 * f], kh[2 * f + 1]);
      aa = make_ulonglong2(ah[2 * f], ah[2 * f + 1]);
    } else {
      ld4x(kp + 4 * (rg + 4 * f), kk.x, kk.y);
      ld4x(ap + 4 * (rg + 4 * f), aa.x, aa.y);
    }
    S[0][2 * f] = mul2(S[0][2 * f], aa.x);
    S[0][2 * f + 1] = mul2(S[0][2 * f + 1], aa.y);
    S[1][2 * f] = mul2(S[1][2 * f], aa.x);
    S[1][2 * f + 1] = mul2(S[1][2 * f + 1], aa.y);
    dA0 = fma2(kk.x, S[0][2 * f], dA0);
    dB0 = fma2(kk.y, S[0][2 * f + 1], dB0);
    dA1 = fma2(kk.x, S[1][2 * f], dA1);
    dB1 = fma2(kk.y, S[1][2 * f + 1], dB1);
  }
  float d0 = __fadd_rn(sum2(dA0), sum2(dB0));
  float d1 = __fadd_rn(sum2(dA1), sum2(dB1));
  d0 = __fadd_rn(d0, __shfl_xor_sync(kFull, d0, 1));
  d1 = __fadd_rn(d1, __shfl_xor_sync(kFull, d1, 1));
  d0 = __fadd_rn(d0, __shfl_xor_sync(kFull, d0, 2));
  d1 = __fadd_rn(d1, __shfl_xor_sync(kFull, d1, 2));
  const float del0 = __fmul_rn(beta, __fsub_rn(v0, d0));
  const float del1 = __fmul_rn(beta, __fsub_rn(v1, d1));
  const f2 D0 = pack2(del0, del0), D1 = pack2(del1, del1);
  f2 oA0 = 0, oB0 = 0, oA1 = 0, oB1 = 0;
#pragma unroll
  for (int f = 0; f < F; ++f) {
    ulonglong2 kk;
    if (HOIST) kk = make_ulonglong2(kh[2 * f], kh[2 * f + 1]);
    else ld4x(kp + 4 * (rg + 4 * f), kk.x, kk.y);
    S[0][2 * f] = fma2(kk.x, D0, S[0][2 * f]);
    S[0][2 * f + 1] = fma2(kk.y, D0, S[0][2 * f + 1]);
    S[1][2 * f] = fma2(kk.x, D1, S[1][2 * f]);
    S[1][2 * f + 1] = fma2(kk.y, D1, S[1][2 * f + 1]);
    if (WANT_O) {
      ulonglong2 qq;
      ld4x(qp + 4 * (rg + 4 * f), qq.x, qq.y);
      oA0 = fma2(qq.x, S[0][2 * f], oA0);
      oB0 = fma2(qq.y, S[0][2 * f + 1], oB0);
      oA1 = fma2(qq.x, S[1][2 * f], oA1);
      oB1 = fma2(qq.y, S[1][2 * f + 1], oB1);
    }
  }
  if (WANT_O) {
    float p0 = sum2(oA0) + sum2(oB0);
    float p1 = sum2(oA1) + sum2(oB1);
    p0 += __shfl_xor_sync(kFull, p0, 1);
    p1 += __shfl_xor_sync(kFull, p1, 1);
    p0 += __shfl_xor_sync(kFull, p0, 2);
    p1 += __shfl_xor_sync(kFull, p1, 2);
    o0 = p0;
    o1 = p1;
  }
}

// The same step with the token's vectors in one record (Rec layout).
template <int D, bool WANT_O, typename Tin, bool HOIST = false>
__device__ __forceinline__ void kda_step(f2 (&S)[2][D / 8], const Tin *rec,
                                         int rg, int j0, float &o0, float &o1) {
  typedef Rec<D, Tin> R;
  kda_step_ptrs<D, WANT_O, Tin, Tin, HOIST>(S, rec + R::kK, rec + R::kA, rec + R::kQ,
                                            rec + R::kV, rec + R::kB, rg, j0, o0, o1);
}

}  // namespace kda
