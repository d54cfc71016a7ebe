// Verify + lazily fused ReplaySSM commit + ordinary decode, one kernel.
// ("ReplaySSM shrinks rollback state" and "Small tensor copies leave the hot
// path", vLLM Kimi K3 optimisation page.)
//
// One CTA owns one (sequence, head) unit for the whole launch, so its state is
// read from HBM once and written at most once:
//   1. the `accepted` ring entries recorded by the last commit are replayed
//      onto the state token by token (kda_step) and the state is written once;
//   2. speculative rows: the T drafted tokens' outputs are computed from the
//      committed state in chunk form (no draft state exists anywhere) and the
//      drafted inputs are copied into the ring;  ordinary rows: the tokens are
//      applied with kda_step and committed.
//
// Thread mapping (head dim D = d_k = d_v): 2*D threads; thread tid owns value
// columns j0 = 2*(tid/4), j0+1 and, of each, key rows c = 4*(rg + 4*i) + e,
// rg = tid % 4, i < D/16, e < 4.  Rows are held as pairs (c, c+1) in 64-bit
// registers and advanced with packed fp32x2 instructions.  The four threads
// of a column reduce with two xor-shuffles.
//
// Chunk form of T drafted tokens from the committed state S (per column j):
//   gamma_t = prod_{r<=t} alpha_r,  kt_t = gamma_t k_t,  qt_t = gamma_t q_t
//   A_ts = sum_c k_tc k_sc gamma_tc / gamma_sc  (s < t)
//   B_ts = sum_c q_tc k_sc gamma_tc / gamma_sc  (s <= t)
//   delta_t = beta_t (v_tj - (S^T kt_t)_j - sum_{s<t} A_ts delta_s)
//   o_tj    = (S^T qt_t)_j + sum_{s<=t} B_ts delta_s
// which is the recurrence unrolled over the drafted tokens.
#include "kda_internal.cuh"

namespace kda {
namespace {

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

// Per-token record in shared memory (fp32): k[D] alpha[D] q[D] v[D] beta pad3.
template <int D>
struct Rec {
  static constexpr int kStride = 4 * D + 4;
  static constexpr int kK = 0, kA = D, kQ = 2 * D, kV = 3 * D, kB = 4 * D;
};

// One token of the recurrence on the thread's slice of S, fixed rounding:
//   S' = Diag(alpha) S;  dot_j = sum_c k_c S'_cj;  delta_j = beta (v_j - dot_j)
//   S  = S' + k delta^T;  o_j = sum_c q_c S_cj  (when WANT_O)
// The only code that advances a committed state: replay, decode and
// materialize all call it, so identical inputs give identical bits.
template <int D, bool WANT_O>
__device__ __forceinline__ void kda_step(f2 (&S)[2][D / 8], const float *rec,
                                         int rg, int j0, float &o0, float &o1) {
  constexpr int F = D / 16;
  const ulonglong2 *k2 = reinterpret_cast<const ulonglong2 *>(rec + Rec<D>::kK);
  const ulonglong2 *a2 = reinterpret_cast<const ulonglong2 *>(rec + Rec<D>::kA);
  const ulonglong2 *q2 = reinterpret_cast<const ulonglong2 *>(rec + Rec<D>::kQ);
  f2 dA0 = 0, dB0 = 0, dA1 = 0, dB1 = 0;
#pragma unroll
  for (int f = 0; f < F; ++f) {
    const ulonglong2 kk = k2[rg + 4 * f];
    const ulonglong2 aa = a2[rg + 4 * f];
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
  const float beta = rec[Rec<D>::kB];
  const float del0 = __fmul_rn(beta, __fsub_rn(rec[Rec<D>::kV + j0], d0));
  const float del1 = __fmul_rn(beta, __fsub_rn(rec[Rec<D>::kV + j0 + 1], d1));
  const f2 D0 = pack2(del0, del0), D1 = pack2(del1, del1);
  f2 oA0 = 0, oB0 = 0, oA1 = 0, oB1 = 0;
#pragma unroll
  for (int f = 0; f < F; ++f) {
    const ulonglong2 kk = k2[rg + 4 * f];
    S[0][2 * f] = fma2(kk.x, D0, S[0][2 * f]);
    S[0][2 * f + 1] = fma2(kk.y, D0, S[0][2 * f + 1]);
    S[1][2 * f] = fma2(kk.x, D1, S[1][2 * f]);
    S[1][2 * f + 1] = fma2(kk.y, D1, S[1][2 * f + 1]);
    if (WANT_O) {
      const ulonglong2 qq = q2[rg + 4 * f];
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

// Raw 16-byte vector of inputs -> fp32 (4 or 8 values).
template <typename Tin>
__device__ __forceinline__ void cvt16(const uint4 &raw, float *dst);
template <>
__device__ __forceinline__ void cvt16<float>(const uint4 &raw, float *dst) {
  *reinterpret_cast<float4 *>(dst) =
      make_float4(__uint_as_float(raw.x), __uint_as_float(raw.y),
                  __uint_as_float(raw.z), __uint_as_float(raw.w));
}
template <>
__device__ __forceinline__ void cvt16<__nv_bfloat16>(const uint4 &raw, float *dst) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
  *reinterpret_cast<float4 *>(dst) =
      make_float4(__uint_as_float(w[0] << 16), __uint_as_float(w[0] & 0xffff0000u),
                  __uint_as_float(w[1] << 16), __uint_as_float(w[1] & 0xffff0000u));
  *reinterpret_cast<float4 *>(dst + 4) =
      make_float4(__uint_as_float(w[2] << 16), __uint_as_float(w[2] & 0xffff0000u),
                  __uint_as_float(w[3] << 16), __uint_as_float(w[3] & 0xffff0000u));
}

// Ring entries to replay (k, alpha, v, beta of `acc` entries) and this
// launch's tokens (k, alpha, v, q, beta of T rows) -> fp32 records in shared
// memory.  Loads are issued in batches of four 16-byte vectors per thread
// before any of them is converted, so their latencies overlap.
template <int D, typename Tin>
__device__ __forceinline__ void load_all_records(
    float *rep, float *drf, int acc, int T, const Tin *rk, const Tin *ra,
    const Tin *rv, const Tin *rb, const Tin *tk, const Tin *ta, const Tin *tv,
    const Tin *tq, const Tin *tb, size_t tok_stride, size_t beta_stride,
    int tid) {
  constexpr int NT = 2 * D;
  constexpr int E = InVec<Tin>::kElems;
  constexpr int CH = D / E;
  constexpr int R = 4;
  const int nring = acc * 3 * CH;
  const int ntot = nring + T * 4 * CH;
  float bval = 0.f;
  float *bdst = nullptr;
  if (tid < acc) {
    bval = in_scalar<Tin>(rb + tid);
    bdst = rep + tid * Rec<D>::kStride + Rec<D>::kB;
  } else if (tid < acc + T) {
    bval = in_scalar<Tin>(tb + (size_t)(tid - acc) * beta_stride);
    bdst = drf + (tid - acc) * Rec<D>::kStride + Rec<D>::kB;
  }
  for (int base = 0; base < ntot; base += R * NT) {
    uint4 buf[R];
    float *dst[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int idx = base + r * NT + tid;
      dst[r] = nullptr;
      if (idx < ntot) {
        const Tin *src;
        if (idx < nring) {
          const int t = idx / (3 * CH), rem = idx - t * 3 * CH;
          const int which = rem / CH, ch = rem - which * CH;
          src = (which == 0 ? rk : which == 1 ? ra : rv) + t * D + ch * E;
          dst[r] = rep + t * Rec<D>::kStride +
                   (which == 0 ? Rec<D>::kK : which == 1 ? Rec<D>::kA : Rec<D>::kV) + ch * E;
        } else {
          const int j = idx - nring;
          const int t = j / (4 * CH), rem = j - t * 4 * CH;
          const int which = rem / CH, ch = rem - which * CH;
          src = (which == 0 ? tk : which == 1 ? ta : which == 2 ? tv : tq) +
                (size_t)t * tok_stride + ch * E;
          dst[r] = drf + t * Rec<D>::kStride +
                   (which == 0 ? Rec<D>::kK : which == 1 ? Rec<D>::kA
                    : which == 2 ? Rec<D>::kV : Rec<D>::kQ) + ch * E;
        }
        buf[r] = *reinterpret_cast<const uint4 *>(src);
      }
    }
#pragma unroll
    for (int r = 0; r < R; ++r)
      if (dst[r]) cvt16<Tin>(buf[r], dst[r]);
  }
  if (bdst) *bdst = bval;
}

// Shared-memory carve-up (floats) for a launch with ring depth `depth` and at
// most `maxT` tokens per row: replay records, token records, kt, qt, kh, the
// reduced dots xs / ys, and the kTMax x kTMax matrices A and B.
template <int D>
struct Smem {
  int rep, drf, kt, qt, kh, xs, ys, am, bm, total;
  __host__ __device__ Smem(int depth, int maxT) {
    rep = 0;
    drf = rep + depth * Rec<D>::kStride;
    kt = drf + maxT * Rec<D>::kStride;
    qt = kt + maxT * D;
    kh = qt + maxT * D;
    xs = kh + maxT * D;
    ys = xs + maxT * D;
    am = ys + maxT * D;
    bm = am + kTMax * kTMax;
    total = bm + kTMax * kTMax;
  }
};

// Per-launch shared quantities of the chunk form (independent of S):
// kt, qt (gamma-scaled), A (without beta) and B.
template <int D>
__device__ void draft_prep(float *sm, const Smem<D> &L, int T, int tid) {
  constexpr int NT = 2 * D;
  const float *rec = sm + L.drf;
  float *kt = sm + L.kt, *qt = sm + L.qt, *kh = sm + L.kh;
  int unsafe = 0;
  for (int c = tid; c < D; c += NT) {
    float g = 1.f;
    for (int t = 0; t < T; ++t) {
      const float *r = rec + t * Rec<D>::kStride;
      g = g * r[Rec<D>::kA + c];
      kt[t * D + c] = g * r[Rec<D>::kK + c];
      qt[t * D + c] = g * r[Rec<D>::kQ + c];
      unsafe |= !(g >= 0x1p-60f && g <= 0x1p60f);
      kh[t * D + c] = r[Rec<D>::kK + c] * __frcp_rn(g);
    }
  }
  unsafe = __syncthreads_or(unsafe);
  // T^2 pair dots (B: s <= t, then A: s < t), 4 lanes per pair, each lane a
  // quarter of the key channels (interleaved float4 groups).
  const int nb = T * (T + 1) / 2, npairs = T * T;
  const int rg = tid & 3;
  for (int base = 0; base < npairs * 4; base += NT) {
    const int item = base + tid;
    const int pair = item >> 2;
    float acc = 0.f;
    int t = 0, s = 0;
    const bool valid = pair < npairs;
    const bool isB = pair < nb;
    if (valid) {
      int r = isB ? pair : pair - nb;
      if (isB) {
        while (r >= t + 1) { r -= t + 1; ++t; }
        s = r;
      } else {
        t = 1;
        while (r >= t) { r -= t; ++t; }
        s = r;
      }
      if (!unsafe) {
        const float4 *x4 = reinterpret_cast<const float4 *>((isB ? qt : kt) + t * D);
        const float4 *h4 = reinterpret_cast<const float4 *>(kh + s * D);
        for (int m = rg; m < D / 4; m += 4) {
          const float4 x = x4[m], y = h4[m];
          acc = fmaf(x.x, y.x, fmaf(x.y, y.y, fmaf(x.z, y.z, fmaf(x.w, y.w, acc))));
        }
      } else {
        // decay products taken explicitly when gamma leaves the safe range
        for (int c = rg; c < D; c += 4) {
          float pr = 1.f;
          for (int u = s + 1; u <= t; ++u) pr *= rec[u * Rec<D>::kStride + Rec<D>::kA + c];
          const float x = rec[t * Rec<D>::kStride + (isB ? Rec<D>::kQ : Rec<D>::kK) + c];
          acc = fmaf(x * rec[s * Rec<D>::kStride + Rec<D>::kK + c], pr, acc);
        }
      }
    }
    acc += __shfl_xor_sync(kFull, acc, 1);
    acc += __shfl_xor_sync(kFull, acc, 2);
    if (valid && rg == 0) {
      if (isB) sm[L.bm + t * kTMax + s] = acc;
      else sm[L.am + t * kTMax + s] = acc;
    }
  }
}

template <int D, typename Tin>
__global__ void __launch_bounds__(2 * D, 2)
    verify_kernel(const VerifyParams p) {
  constexpr int NT = 2 * D;
  constexpr int F = D / 16;
  extern __shared__ float4 smem4[];
  float *sm = reinterpret_cast<float *>(smem4);
  __shared__ int s_info[6];  // skip, slot, accepted, T, tok0, spec

  const int h = blockIdx.x;
  const int i = blockIdx.y;
  const int tid = threadIdx.x;
  const int H = p.H;
  const Smem<D> L(p.depth, p.max_T);
  const int rg = tid & 3;
  const int j0 = 2 * (tid >> 2);

  // 1. the unit's state -> registers first (its address needs only the slot
  //    id), 16-byte loads, 4 lanes cover 64 contiguous bytes of a column.
  const int slot0 = p.state_slots[i];
  const bool slot_ok = slot0 >= 0 && slot0 < p.P;
  float *st = p.pool + ((size_t)(slot_ok ? slot0 : 0) * H + h) * D * D;
  f2 S[2][2 * F];
  if (slot_ok) {
    const ulonglong2 *c0 = reinterpret_cast<const ulonglong2 *>(st + (size_t)j0 * D);
    const ulonglong2 *c1 = c0 + D / 4;
#pragma unroll
    for (int f = 0; f < F; ++f) {
      const ulonglong2 x = c0[rg + 4 * f];
      const ulonglong2 y = c1[rg + 4 * f];
      S[0][2 * f] = x.x; S[0][2 * f + 1] = x.y;
      S[1][2 * f] = y.x; S[1][2 * f + 1] = y.y;
    }
  }
  // later-wave units' states -> L2 now, so HBM streams while this wave computes
  if (tid == 32 && p.prefetch_stride > 0) {
    const int b = i * H + h;
    if (b < p.prefetch_stride) {
      for (int u = b + p.prefetch_stride; u < p.B * H; u += p.prefetch_stride) {
        const int su = p.state_slots[u / H];
        if (su >= 0 && su < p.P) {
          const float *pu = p.pool + ((size_t)su * H + (u - (u / H) * H)) * D * D;
          asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;"
                       :: "l"(pu), "r"(D * D * 4) : "memory");
        }
      }
    }
  }
  if (tid == 0) {
    int skip = 0, acc = 0, T = 0, tok0 = 0, spec = 0;
    if (!slot_ok) {
      set_error(p.err, KDA_DERR_SLOT);
      skip = 1;
    }
    if (!skip && p.mode == 0) {
      const int c0 = p.cu_seqlens[i], c1 = p.cu_seqlens[i + 1];
      if (c0 < 0 || c1 < c0 || c1 > p.N) {
        set_error(p.err, KDA_DERR_SEGMENT);
        skip = 1;
      } else {
        tok0 = c0;
        T = c1 - c0;
        spec = p.is_spec ? (p.is_spec[i] != 0) : 1;
        if (T > p.max_T || (spec && T > p.depth)) {
          set_error(p.err, KDA_DERR_DEPTH);
          skip = 1;
        }
      }
    }
    if (!skip) {
      const int32_t *c = p.ctrl + ((size_t)slot0 * H + h) * 2;
      const int pend = c[0];
      acc = c[1];
      if (pend < 0 || pend > p.depth || acc < 0 || acc > pend) {
        set_error(p.err, KDA_DERR_RING);
        skip = 1;
      }
    }
    s_info[0] = skip; s_info[1] = slot0; s_info[2] = acc;
    s_info[3] = T; s_info[4] = tok0; s_info[5] = spec;
  }
  __syncthreads();
  if (s_info[0]) return;
  const int slot = s_info[1], acc = s_info[2], T = s_info[3];
  const int tok0 = s_info[4];
  const bool spec = s_info[5] != 0;

  // 2. ring entries to replay and this launch's tokens -> shared memory
  const size_t unit = (size_t)slot * H + h;
  float *tsm = sm + L.drf;
  {
    const size_t row = (size_t)tok0 * H + h;
    const Tin *tq = reinterpret_cast<const Tin *>(p.q);
    const Tin *tk = reinterpret_cast<const Tin *>(p.k);
    const Tin *tv = reinterpret_cast<const Tin *>(p.v);
    const Tin *ta = reinterpret_cast<const Tin *>(p.alpha);
    const Tin *tbe = reinterpret_cast<const Tin *>(p.beta);
    load_all_records<D, Tin>(
        sm + L.rep, tsm, acc, T,
        reinterpret_cast<const Tin *>(p.rk) + unit * p.depth * D,
        reinterpret_cast<const Tin *>(p.ra) + unit * p.depth * D,
        reinterpret_cast<const Tin *>(p.rv) + unit * p.depth * D,
        reinterpret_cast<const Tin *>(p.rb) + unit * p.depth,
        tk ? tk + row * D : nullptr, ta ? ta + row * D : nullptr,
        tv ? tv + row * D : nullptr, tq ? tq + row * D : nullptr,
        tbe ? tbe + row : nullptr, (size_t)H * D, (size_t)H, tid);
  }
  __syncthreads();
  // chunk-form quantities of the drafts (do not depend on S; overlap the loads)
  if (spec && T > 0) {
    draft_prep<D>(sm, L, T, tid);
    __syncthreads();
  }

  // 3. lazy commit: replay the accepted entries
  float o0 = 0.f, o1 = 0.f;
  for (int t = 0; t < acc; ++t)
    kda_step<D, false>(S, sm + L.rep + t * Rec<D>::kStride, rg, j0, o0, o1);

  auto store_state = [&]() {
    ulonglong2 *c0 = reinterpret_cast<ulonglong2 *>(st + (size_t)j0 * D);
    ulonglong2 *c1 = c0 + D / 4;
#pragma unroll
    for (int f = 0; f < F; ++f) {
      c0[rg + 4 * f] = make_ulonglong2(S[0][2 * f], S[0][2 * f + 1]);
      c1[rg + 4 * f] = make_ulonglong2(S[1][2 * f], S[1][2 * f + 1]);
    }
  };

  if (!spec) {
    // ordinary decode (or materialize): apply and commit
    for (int t = 0; t < T; ++t) {
      kda_step<D, true>(S, tsm + t * Rec<D>::kStride, rg, j0, o0, o1);
      if (rg == 0)
        *reinterpret_cast<float2 *>(p.o + ((size_t)(tok0 + t) * H + h) * D + j0) =
            make_float2(o0, o1);
    }
    if (acc > 0 || T > 0) store_state();
    if (tid == 0) {
      int32_t *c = p.ctrl + unit * 2;
      c[0] = 0;
      c[1] = 0;
    }
    return;
  }

  if (acc > 0) store_state();
  // ring <- this launch's drafted inputs (the replayed entries are in smem)
  {
    constexpr int E = InVec<Tin>::kElems;
    constexpr int CH = D / E;
    Tin *wk = reinterpret_cast<Tin *>(p.rk) + unit * p.depth * D;
    Tin *wa = reinterpret_cast<Tin *>(p.ra) + unit * p.depth * D;
    Tin *wv = reinterpret_cast<Tin *>(p.rv) + unit * p.depth * D;
    Tin *wb = reinterpret_cast<Tin *>(p.rb) + unit * p.depth;
    for (int idx = tid; idx < T * 3 * CH; idx += NT) {
      const int t = idx / (3 * CH);
      const int r = idx - t * 3 * CH;
      const int which = r / CH, ch = r - (r / CH) * CH;
      const int off = which == 0 ? Rec<D>::kK : which == 1 ? Rec<D>::kA : Rec<D>::kV;
      Tin *dst = (which == 0 ? wk : which == 1 ? wa : wv) + (size_t)t * D + ch * E;
      InVec<Tin>::store(dst, tsm + t * Rec<D>::kStride + off + ch * E);
    }
    for (int t = tid; t < T; t += NT)
      out_scalar<Tin>(wb + t, tsm[t * Rec<D>::kStride + Rec<D>::kB]);
  }
  if (tid == 0) {
    int32_t *c = p.ctrl + unit * 2;
    c[0] = T;
    c[1] = 0;
  }

  // 4. drafts: (S^T kt_t, S^T qt_t) for the thread's two columns, four
  //    drafted tokens per pass, then a column-wise triangular solve.
  const float *kt = sm + L.kt;
  const float *qt = sm + L.qt;
  float *xs = sm + L.xs;
  float *ys = sm + L.ys;
  for (int t0 = 0; t0 < T; t0 += 4) {
    f2 ak[4][2], aq[4][2];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      ak[u][0] = ak[u][1] = aq[u][0] = aq[u][1] = 0;
#pragma unroll
    for (int f = 0; f < F; ++f) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (t0 + u < T) {
          const ulonglong2 kk =
              reinterpret_cast<const ulonglong2 *>(kt + (t0 + u) * D)[rg + 4 * f];
          const ulonglong2 qq =
              reinterpret_cast<const ulonglong2 *>(qt + (t0 + u) * D)[rg + 4 * f];
          ak[u][0] = fma2(kk.x, S[0][2 * f], ak[u][0]);
          ak[u][0] = fma2(kk.y, S[0][2 * f + 1], ak[u][0]);
          ak[u][1] = fma2(kk.x, S[1][2 * f], ak[u][1]);
          ak[u][1] = fma2(kk.y, S[1][2 * f + 1], ak[u][1]);
          aq[u][0] = fma2(qq.x, S[0][2 * f], aq[u][0]);
          aq[u][0] = fma2(qq.y, S[0][2 * f + 1], aq[u][0]);
          aq[u][1] = fma2(qq.x, S[1][2 * f], aq[u][1]);
          aq[u][1] = fma2(qq.y, S[1][2 * f + 1], aq[u][1]);
        }
      }
    }
    // reduce the 16 partial dots (4 tokens x {x0, x1, y0, y1}) over the four
    // row groups of the column pair; lane rg ends with token t0 + rg.
    {
      float v[4][4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        v[u][0] = sum2(ak[u][0]);
        v[u][1] = sum2(ak[u][1]);
        v[u][2] = sum2(aq[u][0]);
        v[u][3] = sum2(aq[u][1]);
      }
      const bool hi2 = (rg & 2) != 0, hi1 = (rg & 1) != 0;
      float r[2][4];
#pragma unroll
      for (int u = 0; u < 2; ++u)
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const float keep = hi2 ? v[u + 2][w] : v[u][w];
          const float give = hi2 ? v[u][w] : v[u + 2][w];
          r[u][w] = keep + __shfl_xor_sync(kFull, give, 2);
        }
      float fin[4];
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const float keep = hi1 ? r[1][w] : r[0][w];
        const float give = hi1 ? r[0][w] : r[1][w];
        fin[w] = keep + __shfl_xor_sync(kFull, give, 1);
      }
      const int t = t0 + rg;
      if (t < T) {
        *reinterpret_cast<float2 *>(xs + t * D + j0) = make_float2(fin[0], fin[1]);
        *reinterpret_cast<float2 *>(ys + t * D + j0) = make_float2(fin[2], fin[3]);
      }
    }
  }
  __syncthreads();
  // column-wise forward substitution: thread -> (column, parity of t)
  {
    const int j = tid >> 1, par = tid & 1;
    const float *am = sm + L.am, *bm = sm + L.bm;
    float del[kTMax];
#pragma unroll
    for (int t = 0; t < kTMax; ++t) {
      if (t < T) {
        const float *r = tsm + t * Rec<D>::kStride;
        float a = xs[t * D + j];
#pragma unroll
        for (int s = 0; s < t; ++s) a = fmaf(am[t * kTMax + s], del[s], a);
        del[t] = r[Rec<D>::kB] * (r[Rec<D>::kV + j] - a);
      }
    }
#pragma unroll
    for (int t = 0; t < kTMax; ++t) {
      if (t < T && (t & 1) == par) {
        float o = ys[t * D + j];
#pragma unroll
        for (int s = 0; s <= t; ++s) o = fmaf(bm[t * kTMax + s], del[s], o);
        p.o[((size_t)(tok0 + t) * H + h) * D + j] = o;
      }
    }
  }
}

__global__ void commit_kernel(const CommitParams p) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= p.B * p.H) return;
  const int i = idx / p.H, h = idx - (idx / p.H) * p.H;
  const int slot = p.slots[i];
  if (slot < 0 || slot >= p.P) {
    set_error(p.err, KDA_DERR_SLOT);
    return;
  }
  int32_t *c = p.ctrl + ((size_t)slot * p.H + h) * 2;
  const int a = p.accepted_len[i];
  if (a < 0 || a > c[0]) {
    set_error(p.err, KDA_DERR_ACCEPT);
    return;
  }
  c[1] = a;
}

__global__ void commit_layers_kernel(const CommitLayersParams p) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= p.B * p.H * p.L) return;
  const int l = idx / (p.B * p.H);
  const int r = idx - l * p.B * p.H;
  const int i = r / p.H, h = r - (r / p.H) * p.H;
  const int slot = p.slots[i];
  if (slot < 0 || slot >= p.P) {
    set_error(p.err, KDA_DERR_SLOT);
    return;
  }
  int32_t *c = p.ctrl[l] + ((size_t)slot * p.H + h) * 2;
  const int a = p.accepted_len[i];
  if (a < 0 || a > c[0]) {
    set_error(p.err, KDA_DERR_ACCEPT);
    return;
  }
  c[1] = a;
}

__global__ void ring_reset_kernel(const CommitParams p) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= p.B * p.H) return;
  const int i = idx / p.H, h = idx - (idx / p.H) * p.H;
  const int slot = p.slots[i];
  if (slot < 0 || slot >= p.P) {
    set_error(p.err, KDA_DERR_SLOT);
    return;
  }
  int32_t *c = p.ctrl + ((size_t)slot * p.H + h) * 2;
  c[0] = 0;
  c[1] = 0;
}

template <int D, typename Tin>
cudaError_t launch_verify_t(VerifyParams p, cudaStream_t s) {
  const size_t smem = verify_smem_bytes(D, p.depth, p.max_T);
  auto kern = verify_kernel<D, Tin>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(
        kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  // CTAs resident in the first wave: they prefetch the later waves' states.
  int dev = 0, sms = 0, per_sm = 0;
  if (cudaGetDevice(&dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 2 * D, smem) ==
          cudaSuccess)
    p.prefetch_stride = per_sm * sms;
  else
    p.prefetch_stride = 0;
  dim3 grid(p.H, p.B);
  kern<<<grid, 2 * D, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

size_t verify_smem_bytes(int D, int depth, int max_T) {
  switch (D) {
    case 16: return sizeof(float) * Smem<16>(depth, max_T).total;
    case 32: return sizeof(float) * Smem<32>(depth, max_T).total;
    case 64: return sizeof(float) * Smem<64>(depth, max_T).total;
    case 128: return sizeof(float) * Smem<128>(depth, max_T).total;
    default: return 0;
  }
}

int verify_max_spec_tokens() { return kTMax; }

cudaError_t launch_verify(const VerifyParams &p, kda_dtype dt, int D,
                          cudaStream_t s) {
  if (p.B == 0) return cudaSuccess;
#define KDA_V(DD)                                                          \
  case DD:                                                                 \
    return dt == KDA_BF16 ? launch_verify_t<DD, __nv_bfloat16>(p, s)       \
                          : launch_verify_t<DD, float>(p, s);
  switch (D) {
    KDA_V(16)
    KDA_V(32)
    KDA_V(64)
    KDA_V(128)
    default:
      return cudaErrorInvalidValue;
  }
#undef KDA_V
}

cudaError_t launch_commit(const CommitParams &p, cudaStream_t s) {
  const int n = p.B * p.H;
  if (n == 0) return cudaSuccess;
  commit_kernel<<<(n + 255) / 256, 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_commit_layers(const CommitLayersParams &p, cudaStream_t s) {
  const int n = p.B * p.H * p.L;
  if (n == 0) return cudaSuccess;
  commit_layers_kernel<<<(n + 255) / 256, 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_ring_reset(const CommitParams &p, cudaStream_t s) {
  const int n = p.B * p.H;
  if (n == 0) return cudaSuccess;
  ring_reset_kernel<<<(n + 255) / 256, 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace kda
