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
#include <mutex>

#include "kda_internal.cuh"
#include "kda_step.cuh"
#include "kda_umma.cuh"

namespace kda {
namespace {

// Ring entries to replay (k, alpha, v, beta of `acc` entries) and this
// launch's tokens (k, alpha, v, q, beta of T rows) -> records in shared
// memory, copied as they are.  Vector rows are numbered ring-first (3 per
// entry) then token rows (4 per token); thread tid always copies 16-byte
// chunk tid % CH of rows tid / CH, + NT / CH, ...  All of a thread's loads
// are issued before any of them is stored.
template <int D, typename Tin>
__device__ __forceinline__ void load_all_records(
    Tin *rep, Tin *drf, int acc, int T, const Tin *rk, const Tin *ra,
    const Tin *rv, const Tin *rb, const Tin *tk, const Tin *ta, const Tin *tv,
    const Tin *tq, const Tin *tb, size_t tok_stride, size_t beta_stride,
    int tid) {
  typedef Rec<D, Tin> RC;
  constexpr int NT = 2 * D;
  constexpr int E = InVec<Tin>::kElems;
  constexpr int CH = D / E;         // power of two
  constexpr int RSTEP = NT / CH;    // vector rows per pass
  constexpr int R = 4;              // loads in flight per thread
  const int ch = tid % CH;
  const int nring = acc * 3, nrows = nring + T * 4;
  Tin bval;
  Tin *bdst = nullptr;
  if (tid < acc) {
    bval = rb[tid];
    bdst = rep + tid * RC::kStride + RC::kB;
  } else if (tid < acc + T) {
    bval = tb[(size_t)(tid - acc) * beta_stride];
    bdst = drf + (tid - acc) * RC::kStride + RC::kB;
  }
  for (int base = tid / CH; base < nrows; base += R * RSTEP) {
    uint4 buf[R];
    Tin *dst[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int row = base + r * RSTEP;
      dst[r] = nullptr;
      if (row < nrows) {
        const Tin *src;
        if (row < nring) {
          const int t = row / 3, which = row - 3 * (row / 3);
          src = (which == 0 ? rk : which == 1 ? ra : rv) + t * D + ch * E;
          dst[r] = rep + t * RC::kStride +
                   (which == 0 ? RC::kK : which == 1 ? RC::kA : RC::kV) + ch * E;
        } else {
          const int rr = row - nring;
          const int t = rr >> 2, which = rr & 3;
          const Tin *base_ptr = which == 0 ? tk : which == 1 ? ta : which == 2 ? tv : tq;
          src = base_ptr + (size_t)t * tok_stride + ch * E;
          dst[r] = drf + t * RC::kStride +
                   (which == 0 ? RC::kK : which == 1 ? RC::kA
                    : which == 2 ? RC::kV : RC::kQ) + ch * E;
        }
        buf[r] = *reinterpret_cast<const uint4 *>(src);
      }
    }
#pragma unroll
    for (int r = 0; r < R; ++r)
      if (dst[r]) *reinterpret_cast<uint4 *>(dst[r]) = buf[r];
  }
  if (bdst) *bdst = bval;
}

// Shared-memory carve-up (bytes from a 1024-byte aligned base) for ring depth
// `depth` and at most `maxT` tokens per row; TP = padded draft count (8 or
// 16).
//   a    tcgen05 A tiles: the committed state as bf16 hi, then lo, K-major
//        128B-swizzled (128 rows = value columns j, K = key rows c);
//   rep  the ring entries to replay;  drf  this launch's token records (both
//        in the input dtype);
//   rb   the bf16 B tile [K~_hi, Q~_hi, K~_lo, Q~_lo] (4 TP rows, K-major
//        128B-swizzled), then (kx) K~ and Q~ in fp32, row-major [2 TP][D];
//   kh = k / gamma;  vb = v and beta of the drafted tokens;  am, bm = the
//   T x T matrices of the triangular solve.
// Nothing of the drafts shares space with the replay records, so the drafts'
// state-independent parts run before the replay.
template <int D, typename Tin>
struct Smem {
  int tp, a, rep, drf, rb, kx, kh, vb, am, bm, total;
  __host__ __device__ Smem(int depth, int maxT) {
    tp = maxT <= 8 ? 8 : 16;
    const int kblk = (D + 63) / 64;  // bf16 K blocks
    a = 0;
    rep = 2 * kblk * 128 * 128;
    drf = rep + depth * Rec<D, Tin>::kBytes;
    rb = (drf + maxT * Rec<D, Tin>::kBytes + 1023) & ~1023;
    kx = rb + kblk * 4 * tp * 128;
    kh = kx + 2 * tp * D * 4;
    vb = kh + tp * D * 4;
    am = vb + (tp * D + tp) * 4;
    bm = am + kTMax * kTMax * 4;
    total = bm + kTMax * kTMax * 4 + 1024;  // + alignment slack
  }
};

// Chunk-form quantities of the drafts that do not depend on S, part 1: one
// thread per (4 key channels, drafted row t): gamma_t = prod_{r<=t} alpha_r,
// the bf16 B tile rows t, TP+t (gamma k, gamma q rounded to bf16) and 2TP+t,
// 3TP+t (the remainders, rounded to bf16), zero rows past T, the fp32 values
// (kx), kh = k / gamma, and v, beta.  Returns whether
// gamma left [2^-60, 2^60] anywhere (then A and B use explicit products).
template <int D, int TP, typename Tin>
__device__ __forceinline__ int prep_tiles(unsigned char *smb, const Smem<D, Tin> &L,
                                          const Tin *drf, int T, int tid) {
  typedef Rec<D, Tin> R;
  constexpr int NT = 2 * D, N1 = 4 * TP;
  float *kh = reinterpret_cast<float *>(smb + L.kh);
  float *vb = reinterpret_cast<float *>(smb + L.vb);
  float *kx = reinterpret_cast<float *>(smb + L.kx);
  unsigned char *sb = smb + L.rb;
  int unsafe = 0;
  for (int item = tid; item < (D / 4) * TP; item += NT) {
    const int c4 = item % (D / 4), t = item / (D / 4);
    float4 kt = make_float4(0.f, 0.f, 0.f, 0.f), qt = kt;
    if (t < T) {
      float4 g = ld4f(drf + R::kA + 4 * c4);
#pragma unroll
      for (int r = 1; r < TP; ++r) {
        if (r <= t) {
          const float4 a = ld4f(drf + r * R::kStride + R::kA + 4 * c4);
          g.x *= a.x; g.y *= a.y; g.z *= a.z; g.w *= a.w;
        }
      }
      const Tin *rr = drf + t * R::kStride;
      const float4 k = ld4f(rr + R::kK + 4 * c4);
      const float4 q = ld4f(rr + R::kQ + 4 * c4);
      kt = make_float4(g.x * k.x, g.y * k.y, g.z * k.z, g.w * k.w);
      qt = make_float4(g.x * q.x, g.y * q.y, g.z * q.z, g.w * q.w);
      const float gm = fminf(fminf(g.x, g.y), fminf(g.z, g.w));
      const float gx = fmaxf(fmaxf(g.x, g.y), fmaxf(g.z, g.w));
      unsafe |= !(gm >= 0x1p-60f && gx <= 0x1p60f);
      *reinterpret_cast<float4 *>(kh + t * D + 4 * c4) =
          make_float4(__fdividef(k.x, g.x), __fdividef(k.y, g.y),
                      __fdividef(k.z, g.z), __fdividef(k.w, g.w));
      *reinterpret_cast<float4 *>(vb + t * D + 4 * c4) = ld4f(rr + R::kV + 4 * c4);
      if (c4 == 0) vb[TP * D + t] = in_scalar<Tin>(rr + R::kB);
    }
    *reinterpret_cast<float4 *>(kx + t * D + 4 * c4) = kt;
    *reinterpret_cast<float4 *>(kx + (TP + t) * D + 4 * c4) = qt;
    uint32_t h0, l0, h1, l1;
    umma::split_bf16x2(kt.x, kt.y, h0, l0);
    umma::split_bf16x2(kt.z, kt.w, h1, l1);
    *reinterpret_cast<uint2 *>(sb + umma::sw128_off16(t, 4 * c4, N1)) = make_uint2(h0, h1);
    *reinterpret_cast<uint2 *>(sb + umma::sw128_off16(2 * TP + t, 4 * c4, N1)) =
        make_uint2(l0, l1);
    umma::split_bf16x2(qt.x, qt.y, h0, l0);
    umma::split_bf16x2(qt.z, qt.w, h1, l1);
    *reinterpret_cast<uint2 *>(sb + umma::sw128_off16(TP + t, 4 * c4, N1)) = make_uint2(h0, h1);
    *reinterpret_cast<uint2 *>(sb + umma::sw128_off16(3 * TP + t, 4 * c4, N1)) =
        make_uint2(l0, l1);
  }
  return unsafe;
}

// Part 2: the T^2 pair dots (B: s <= t, then A: s < t; A without beta),
// 4 lanes per pair, each lane a quarter of the key channels.
template <int D, int TP, typename Tin>
__device__ __forceinline__ void prep_pairs(unsigned char *smb,
                                           const Smem<D, Tin> &L, const Tin *drf,
                                           int T, int tid, int unsafe) {
  typedef Rec<D, Tin> R;
  constexpr int NT = 2 * D;
  const float *kh = reinterpret_cast<const float *>(smb + L.kh);
  const float *kx = reinterpret_cast<const float *>(smb + L.kx);
  float *am = reinterpret_cast<float *>(smb + L.am);
  float *bmat = reinterpret_cast<float *>(smb + L.bm);
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
        // gamma k (row t) or gamma q (row TP + t) in fp32
        const float *xr = kx + (isB ? TP + t : t) * D;
        float acc2 = 0.f;
#pragma unroll
        for (int u = 0; u < D / 16; ++u) {
          const int m = rg + 4 * u;
          const float4 x = *reinterpret_cast<const float4 *>(xr + 4 * m);
          const float4 y = *reinterpret_cast<const float4 *>(kh + s * D + 4 * m);
          acc = fmaf(x.x, y.x, acc);
          acc2 = fmaf(x.y, y.y, acc2);
          acc = fmaf(x.z, y.z, acc);
          acc2 = fmaf(x.w, y.w, acc2);
        }
        acc += acc2;
      } else {
        // decay products taken explicitly when gamma leaves the safe range
        for (int c = rg; c < D; c += 4) {
          float pr = 1.f;
          for (int u = s + 1; u <= t; ++u)
            pr *= in_scalar<Tin>(drf + u * R::kStride + R::kA + c);
          const float x = in_scalar<Tin>(drf + t * R::kStride + (isB ? R::kQ : R::kK) + c);
          acc = fmaf(x * in_scalar<Tin>(drf + s * R::kStride + R::kK + c), pr, acc);
        }
      }
    }
    acc += __shfl_xor_sync(kFull, acc, 1);
    acc += __shfl_xor_sync(kFull, acc, 2);
    if (valid && rg == 0) {
      if (isB) bmat[t * kTMax + s] = acc;
      else am[t * kTMax + s] = acc;
    }
  }
}

// Thread's state slice -> A tiles (row j, K = c): hi = rn_bf16(S) at sa and
// lo = rn_bf16(S - hi) one tile further (hi + lo carries 16 significant bits).
template <int D>
__device__ __forceinline__ void write_state_tiles(unsigned char *sa,
                                                  const f2 (&S)[2][D / 8], int rg,
                                                  int j0) {
  constexpr int F = D / 16;
  constexpr uint32_t kLo = ((D + 63) / 64) * 16384;
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int j = j0 + e;
#pragma unroll
    for (int f = 0; f < F; ++f) {
      float x[4];
      asm("mov.b64 {%0, %1}, %2;" : "=f"(x[0]), "=f"(x[1]) : "l"(S[e][2 * f]));
      asm("mov.b64 {%0, %1}, %2;" : "=f"(x[2]), "=f"(x[3]) : "l"(S[e][2 * f + 1]));
      uint32_t h0, l0, h1, l1;
      umma::split_bf16x2(x[0], x[1], h0, l0);
      umma::split_bf16x2(x[2], x[3], h1, l1);
      const uint32_t off = umma::sw128_off16(j, 4 * (rg + 4 * f), 128);
      *reinterpret_cast<uint2 *>(sa + off) = make_uint2(h0, h1);
      *reinterpret_cast<uint2 *>(sa + kLo + off) = make_uint2(l0, l1);
    }
  }
}

// Column j's drafted outputs from the accumulator lane (TMEM address ta):
// x_t = D[t] + D[2TP + t], y_t = D[TP + t] + D[3TP + t];
// delta_t = beta_t (v_tj - x_t - sum_{s<t} A_ts delta_s),
// o_tj = y_t + sum_{s<=t} B_ts delta_s.  Only t with t % ng == grp are
// written.  Every lane of the warp must call this (TMEM load).
template <int D, int TP, typename Tin>
__device__ __forceinline__ void draft_outputs(const VerifyParams &p,
                                              const unsigned char *smb,
                                              const Smem<D, Tin> &L, uint32_t ta,
                                              int j, int grp, int ng, int T,
                                              int tok0, int h) {
  // x_t = D[t] + D[2TP + t] and y_t = D[TP + t] + D[3TP + t], read 8
  // columns at a time to keep few values live
  float x[TP], y[TP];
#pragma unroll
  for (int c8 = 0; c8 < TP; c8 += 8) {
    uint32_t a[8], b[8];
    umma::tmem_ld8_async(ta + c8, a);
    umma::tmem_ld8_async(ta + 2 * TP + c8, b);
    umma::tmem_wait_ld();
#pragma unroll
    for (int m = 0; m < 8; ++m) x[c8 + m] = __uint_as_float(a[m]) + __uint_as_float(b[m]);
    umma::tmem_ld8_async(ta + TP + c8, a);
    umma::tmem_ld8_async(ta + 3 * TP + c8, b);
    umma::tmem_wait_ld();
#pragma unroll
    for (int m = 0; m < 8; ++m) y[c8 + m] = __uint_as_float(a[m]) + __uint_as_float(b[m]);
  }
  if (j >= D) return;
  const float *vb = reinterpret_cast<const float *>(smb + L.vb);
  const float *am = reinterpret_cast<const float *>(smb + L.am);
  const float *bmat = reinterpret_cast<const float *>(smb + L.bm);
  float del[TP];
#pragma unroll
  for (int t = 0; t < TP; ++t) {
    if (t < T) {
      float a = x[t];
#pragma unroll
      for (int s = 0; s < t; ++s) a = fmaf(am[t * kTMax + s], del[s], a);
      del[t] = vb[TP * D + t] * (vb[t * D + j] - a);
    }
  }
#pragma unroll
  for (int t = 0; t < TP; ++t) {
    if (t < T && t % ng == grp) {
      float o = y[t];
#pragma unroll
      for (int s = 0; s <= t; ++s) o = fmaf(bmat[t * kTMax + s], del[s], o);
      p.o[((size_t)(tok0 + t) * p.H + h) * D + j] = o;
    }
  }
}

template <int D, typename Tin, int TP>
__global__ void __launch_bounds__(2 * D, 2)
    verify_kernel(const VerifyParams p) {
  constexpr int F = D / 16;
  extern __shared__ float4 smem4[];
  unsigned char *smb = umma::align1024(smem4);
  __shared__ int s_acc;  // accepted count to replay, -1: ring word invalid
  __shared__ uint64_t s_mbar;
  __shared__ uint32_t s_tmem;

  const int h = blockIdx.x;
  const int i = blockIdx.y;
  const int tid = threadIdx.x;
  const int H = p.H;
  const Smem<D, Tin> L(p.depth, p.max_T);
  typedef Rec<D, Tin> R;
  const int rg = tid & 3;
  const int j0 = 2 * (tid >> 2);

  // Launched as a programmatic dependent of the previous kernel on the
  // stream, this CTA may start while that kernel's last CTAs still run.
  // Until griddepcontrol.wait returns it only issues L2 prefetch hints for
  // this unit's state and ring entries, at the slot the table holds when
  // read: a relaxed read that the previous kernel may still be writing, so
  // a stale value costs only a useless hint, and L2 is the point where the
  // previous kernel's writes become visible, so no stale data is ever used.
  if (tid == 0) {
    int s0;
    asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];"
                 : "=r"(s0) : "l"(p.state_slots + i) : "memory");
    if (s0 >= 0 && s0 < p.P) {
      const size_t u0 = (size_t)s0 * H + h;
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;"
                   :: "l"(p.pool + u0 * D * D), "r"(D * D * 4) : "memory");
      const uint32_t rbytes = (uint32_t)(p.depth * D * sizeof(Tin));
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;"
                   :: "l"(reinterpret_cast<const Tin *>(p.rk) + u0 * p.depth * D),
                      "r"(rbytes) : "memory");
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;"
                   :: "l"(reinterpret_cast<const Tin *>(p.ra) + u0 * p.depth * D),
                      "r"(rbytes) : "memory");
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;"
                   :: "l"(reinterpret_cast<const Tin *>(p.rv) + u0 * p.depth * D),
                      "r"(rbytes) : "memory");
    }
  }
  // the previous kernel has completed and its writes are visible; the next
  // kernel may be scheduled once every CTA of this one has passed here
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // Round trip 1 (all threads, same addresses): slot, segment, row kind.
  const int slot = p.state_slots[i];
  int tok0 = 0, T = 0, spec = 0, bad = 0;
  if (slot < 0 || slot >= p.P) bad = KDA_DERR_SLOT;
  if (p.mode == 0) {
    const int c0 = p.cu_seqlens[i], c1 = p.cu_seqlens[i + 1];
    spec = p.is_spec ? (p.is_spec[i] != 0) : 1;
    if (!bad) {
      if (c0 < 0 || c1 < c0 || c1 > p.N) {
        bad = KDA_DERR_SEGMENT;
      } else {
        tok0 = c0;
        T = c1 - c0;
        if (T > p.max_T || (spec && T > p.depth)) bad = KDA_DERR_DEPTH;
      }
    }
  }
  if (bad) {
    if (tid == 0) set_error(p.err, (unsigned)bad);
    return;
  }
  const bool drafts = spec && T > 0;

  // Round trip 2, all independent: the state (16-byte loads, 4 lanes per 64
  // contiguous bytes of a column), the ring control word, every ring entry
  // (the accepted count is not known yet), and this launch's tokens.
  const size_t unit = (size_t)slot * H + h;
  float *st = p.pool + unit * D * D;
  f2 S[2][2 * F];
  {
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
  // speculative rows with drafts take their tensor-memory columns now, while
  // the state's loads are in flight (an allocation costs the warp about as
  // long as a DRAM round trip)
  if (drafts && tid < 32) umma::tmem_alloc(&s_tmem, (uint32_t)(4 * TP));
  if (tid == 0) {
    const int32_t *c = p.ctrl + unit * 2;
    const int pend = c[0], acc = c[1];
    const bool okc = pend >= 0 && pend <= p.depth && acc >= 0 && acc <= pend;
    if (!okc) set_error(p.err, KDA_DERR_RING);
    s_acc = okc ? acc : -1;
    if (spec && T > 0) umma::mbar_init(&s_mbar, 1);
  }
  Tin *rep = reinterpret_cast<Tin *>(smb + L.rep);
  Tin *drf = reinterpret_cast<Tin *>(smb + L.drf);
  {
    const size_t row = (size_t)tok0 * H + h;
    const Tin *tq = reinterpret_cast<const Tin *>(p.q);
    const Tin *tk = reinterpret_cast<const Tin *>(p.k);
    const Tin *tv = reinterpret_cast<const Tin *>(p.v);
    const Tin *ta = reinterpret_cast<const Tin *>(p.alpha);
    const Tin *tbe = reinterpret_cast<const Tin *>(p.beta);
    load_all_records<D, Tin>(
        rep, drf, p.depth, T,
        reinterpret_cast<const Tin *>(p.rk) + unit * p.depth * D,
        reinterpret_cast<const Tin *>(p.ra) + unit * p.depth * D,
        reinterpret_cast<const Tin *>(p.rv) + unit * p.depth * D,
        reinterpret_cast<const Tin *>(p.rb) + unit * p.depth,
        tk ? tk + row * D : nullptr, ta ? ta + row * D : nullptr,
        tv ? tv + row * D : nullptr, tq ? tq + row * D : nullptr,
        tbe ? tbe + row : nullptr, (size_t)H * D, (size_t)H, tid);
  }
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const int acc = s_acc;
  if (acc < 0) {
    if (drafts && tid < 32) umma::tmem_dealloc(s_tmem, (uint32_t)(4 * TP));
    return;
  }
  // this unit's loads have landed: stream later waves' states into L2 while
  // this wave computes
  if (tid == 32 && p.prefetch_stride > 0) {
    const int b = i * H + h;
    if (b < p.prefetch_stride) {
      for (int u = b + p.prefetch_stride; u < p.B * H; u += p.prefetch_stride) {
        const int su = p.state_slots[u / H];
        if (su >= 0 && su < p.P) {
          const size_t uu = (size_t)su * H + (u - (u / H) * H);
          asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;"
                       :: "l"(p.pool + uu * D * D), "r"(D * D * 4) : "memory");
          // and its ring entries (k, alpha, v)
          const uint32_t rbytes = (uint32_t)(p.depth * D * sizeof(Tin));
          asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;"
                       :: "l"(reinterpret_cast<const Tin *>(p.rk) + uu * p.depth * D),
                          "r"(rbytes) : "memory");
          asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;"
                       :: "l"(reinterpret_cast<const Tin *>(p.ra) + uu * p.depth * D),
                          "r"(rbytes) : "memory");
          asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;"
                       :: "l"(reinterpret_cast<const Tin *>(p.rv) + uu * p.depth * D),
                          "r"(rbytes) : "memory");
        }
      }
    }
  }

  // The drafts' parts that do not depend on the state (decayed keys and
  // queries, the B tile, the T x T pair dots) while the state's loads land.
  int unsafe = 0;
  if (drafts) {
    unsafe = prep_tiles<D, TP, Tin>(smb, L, drf, T, tid);
    unsafe = __syncthreads_or(unsafe);
    prep_pairs<D, TP, Tin>(smb, L, drf, T, tid, unsafe);
  }

  // Lazy commit: replay the accepted entries onto the state.
  float o0 = 0.f, o1 = 0.f;
  for (int t = 0; t < acc; ++t)
    kda_step<D, false, Tin>(S, rep + t * R::kStride, rg, j0, o0, o1);

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
      kda_step<D, true, Tin>(S, drf + t * R::kStride, rg, j0, o0, o1);
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
  if (T == 0) {
    if (acc > 0) store_state();
    if (tid == 0) {
      int32_t *c = p.ctrl + unit * 2;
      c[0] = 0;
      c[1] = 0;
    }
    return;
  }

  // Drafts: X = S^T [K~ | Q~] on the tensor cores, bf16 splits, one round
  // of MMAs into one accumulator:
  //   D  = S_hi [K~_hi Q~_hi K~_lo Q~_lo]^T   (N = 4 TP)
  //   D += S_lo [K~_hi Q~_hi]^T               (N = 2 TP, first columns)
  //   x_t = D[t] + D[2TP + t],  y_t = D[TP + t] + D[3TP + t]
  // i.e. hi*hi + lo*hi + hi*lo of every product.
  constexpr int N1 = 4 * TP, N2 = 2 * TP, NK = D / 16;  // K steps of 16
  constexpr uint32_t kLoA = ((D + 63) / 64) * 16384;     // S_lo tile offset
  unsigned char *sa = smb + L.a;
  write_state_tiles<D>(sa, S, rg, j0);
  umma::fence_smem_to_async();
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tmem = s_tmem;
  const uint32_t a_base = umma::smem_u32(sa), b_base = umma::smem_u32(smb + L.rb);
  if (tid == 0) {
    // descriptors of later K steps differ only in the start address field
    // (16-byte units)
    const uint32_t id1 = umma::idesc_bf16(128, N1), id2 = umma::idesc_bf16(128, N2);
    const uint64_t da = umma::sdesc_sw128(a_base), db = umma::sdesc_sw128(b_base);
#pragma unroll
    for (int s = 0; s < NK; ++s)
      umma::mma_bf16(tmem, da + (((s >> 2) * 16384 + (s & 3) * 32) >> 4),
                     db + (((s >> 2) * N1 * 128 + (s & 3) * 32) >> 4), id1, s > 0 ? 1u : 0u);
#pragma unroll
    for (int s = 0; s < NK; ++s)
      umma::mma_bf16(tmem, da + ((kLoA + (s >> 2) * 16384 + (s & 3) * 32) >> 4),
                     db + (((s >> 2) * N1 * 128 + (s & 3) * 32) >> 4), id2, 1u);
    umma::commit(&s_mbar);
  }
  // overlapped with the MMAs: the committed state, ring append, ring word
  if (acc > 0) store_state();
  {
    constexpr int E = InVec<Tin>::kElems;
    constexpr int CH = D / E;
    Tin *wk = reinterpret_cast<Tin *>(p.rk) + unit * p.depth * D;
    Tin *wa = reinterpret_cast<Tin *>(p.ra) + unit * p.depth * D;
    Tin *wv = reinterpret_cast<Tin *>(p.rv) + unit * p.depth * D;
    Tin *wb = reinterpret_cast<Tin *>(p.rb) + unit * p.depth;
    // warp 0 issues the MMAs; the others copy
    constexpr int base = 2 * D > 64 ? 32 : 0;
    for (int idx = tid - base; idx >= 0 && idx < T * 3 * CH; idx += 2 * D - base) {
      const int t = idx / (3 * CH);
      const int r = idx - t * 3 * CH;
      const int which = r / CH, ch = r - (r / CH) * CH;
      const int off = which == 0 ? R::kK : which == 1 ? R::kA : R::kV;
      Tin *dst = (which == 0 ? wk : which == 1 ? wa : wv) + (size_t)t * D + ch * E;
      *reinterpret_cast<uint4 *>(dst) =
          *reinterpret_cast<const uint4 *>(drf + t * R::kStride + off + ch * E);
    }
    if (tid - base >= 0 && tid - base < T)
      wb[tid - base] = drf[(tid - base) * R::kStride + R::kB];
    if (tid == base) {
      int32_t *c = p.ctrl + unit * 2;
      c[0] = T;
      c[1] = 0;
    }
  }
  // one thread waits on the tensor cores; the others park on the barrier
  bool ok = tid == 0 ? umma::mbar_wait(&s_mbar, 0, p.spin_limit) : true;
  ok = __syncthreads_and(ok);
  const int waiting = 0;  // the phase still owed by the tensor cores
  umma::fence_after_sync();
  if (!ok) {
    if (tid == 0) {
      set_error(p.err, KDA_DERR_TIMEOUT);
      // give the tensor cores one more bounded chance before TMEM is freed
      if (!umma::mbar_wait(&s_mbar, (uint32_t)waiting, kDrainWaitPolls))
        set_error(p.err, KDA_DERR_UNSAFE);
    }
  } else {
    // One thread per value column: triangular solve and outputs.  Warp w
    // can read only TMEM lanes 32 (w % 4) .. 32 (w % 4) + 31 (value columns);
    // the NT / 128 groups of four warps each repeat the solve and write the
    // drafted positions t with t % groups == group.
    const int w = tid >> 5, q = w & 3;
    if (32 * q < D) {
      const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16);
      const int ng = D >= 64 ? D / 64 : 1;  // (2 D threads) / 128
      draft_outputs<D, TP, Tin>(p, smb, L, ta, (q << 5) + (tid & 31), w >> 2, ng, T,
                                tok0, h);
    }
  }
  umma::fence_before_sync();
  __syncthreads();
  if (tid < 32) umma::tmem_dealloc(tmem, (uint32_t)N1);
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

// ---------------------------------------------------------------------------
// Direct per-position snapshots, the design that ReplaySSM replaces ("ReplaySSM
// shrinks rollback state": a direct implementation stores the state at every
// drafted position, T extra state writes per step).  Kept as the ablation
// baseline.  One CTA per (sequence, head) with the thread mapping of
// verify_kernel; every drafted token is applied with kda_step and the state
// after token t is written to snapshot t, so snapshot a - 1 holds the same
// bits as the state a ReplaySSM commit of a tokens rebuilds.
template <int D, typename Tin>
__global__ void __launch_bounds__(2 * D, 2)
    verify_snapshot_kernel(const SnapshotParams p) {
  constexpr int F = D / 16;
  typedef Rec<D, Tin> R;
  extern __shared__ float4 smem4[];
  Tin *drf = reinterpret_cast<Tin *>(smem4);
  const int h = blockIdx.x, i = blockIdx.y, tid = threadIdx.x, H = p.H;
  const int rg = tid & 3, j0 = 2 * (tid >> 2);
  const int slot = p.state_slots[i];
  const int c0 = p.cu_seqlens[i], c1 = p.cu_seqlens[i + 1];
  int bad = 0;
  if (slot < 0 || slot >= p.P) bad = KDA_DERR_SLOT;
  else if (c0 < 0 || c1 < c0 || c1 > p.N) bad = KDA_DERR_SEGMENT;
  else if (c1 - c0 > p.max_T) bad = KDA_DERR_DEPTH;
  if (bad) {
    if (tid == 0) set_error(p.err, (unsigned)bad);
    return;
  }
  const int T = c1 - c0;
  const float *st = p.pool + ((size_t)slot * H + h) * D * D;
  f2 S[2][2 * F];
  {
    const ulonglong2 *a0 = reinterpret_cast<const ulonglong2 *>(st + (size_t)j0 * D);
    const ulonglong2 *a1 = a0 + D / 4;
#pragma unroll
    for (int f = 0; f < F; ++f) {
      const ulonglong2 x = a0[rg + 4 * f];
      const ulonglong2 y = a1[rg + 4 * f];
      S[0][2 * f] = x.x; S[0][2 * f + 1] = x.y;
      S[1][2 * f] = y.x; S[1][2 * f + 1] = y.y;
    }
  }
  if (T > 0) {
    const size_t row = (size_t)c0 * H + h;
    load_all_records<D, Tin>(
        nullptr, drf, 0, T, nullptr, nullptr, nullptr, nullptr,
        reinterpret_cast<const Tin *>(p.k) + row * D,
        reinterpret_cast<const Tin *>(p.alpha) + row * D,
        reinterpret_cast<const Tin *>(p.v) + row * D,
        reinterpret_cast<const Tin *>(p.q) + row * D,
        reinterpret_cast<const Tin *>(p.beta) + row, (size_t)H * D, (size_t)H, tid);
  }
  __syncthreads();
  float o0 = 0.f, o1 = 0.f;
  for (int t = 0; t < T; ++t) {
    kda_step<D, true, Tin>(S, drf + t * R::kStride, rg, j0, o0, o1);
    if (rg == 0)
      *reinterpret_cast<float2 *>(p.o + ((size_t)(c0 + t) * H + h) * D + j0) =
          make_float2(o0, o1);
    float *sn = p.snap + (((size_t)i * p.max_T + t) * H + h) * D * D;
    ulonglong2 *w0 = reinterpret_cast<ulonglong2 *>(sn + (size_t)j0 * D);
    ulonglong2 *w1 = w0 + D / 4;
#pragma unroll
    for (int f = 0; f < F; ++f) {
      w0[rg + 4 * f] = make_ulonglong2(S[0][2 * f], S[0][2 * f + 1]);
      w1[rg + 4 * f] = make_ulonglong2(S[1][2 * f], S[1][2 * f + 1]);
    }
  }
}

// Commit of the direct design: pool(slot, h) = snapshot accepted_len - 1 of
// its row (a plain copy; nothing when 0 tokens were accepted).  One CTA per
// (sequence, head), every thread's loads issued before its stores.
template <int D>
__global__ void __launch_bounds__(256) commit_snapshot_kernel(const SnapshotParams p) {
  constexpr int N4 = D * D / 4;
  constexpr int PER = (N4 + 255) / 256;
  const int h = blockIdx.x, i = blockIdx.y, tid = threadIdx.x, H = p.H;
  const int a = p.accepted_len[i];
  const int slot = p.state_slots[i];
  if (a < 0 || a > p.max_T) {
    if (tid == 0) set_error(p.err, KDA_DERR_ACCEPT);
    return;
  }
  if (slot < 0 || slot >= p.P) {
    if (tid == 0) set_error(p.err, KDA_DERR_SLOT);
    return;
  }
  if (a == 0) return;
  const float4 *src = reinterpret_cast<const float4 *>(
      p.snap + (((size_t)i * p.max_T + (a - 1)) * H + h) * D * D);
  float4 *dst = reinterpret_cast<float4 *>(p.pool + ((size_t)slot * H + h) * D * D);
  float4 buf[PER];
#pragma unroll
  for (int r = 0; r < PER; ++r)
    if (tid + 256 * r < N4) buf[r] = src[tid + 256 * r];
#pragma unroll
  for (int r = 0; r < PER; ++r)
    if (tid + 256 * r < N4) dst[tid + 256 * r] = buf[r];
}

// CTAs of `kern` that fit on one SM at once: the shared-memory, register
// and thread limits of the device against the kernel's needs (taken as the
// larger of this and the runtime's occupancy answer, which can assume a
// smaller shared-memory carveout than the launch gets).  0 if unknown.
int resident_ctas(const void *kern, int threads, size_t dyn_smem) {
  int dev = 0, smem_sm = 0, regs_sm = 0, thr_sm = 0, reserved = 0, api = 0;
  cudaFuncAttributes fa;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaFuncGetAttributes(&fa, kern) != cudaSuccess ||
      cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) !=
          cudaSuccess ||
      cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev) !=
          cudaSuccess ||
      cudaDeviceGetAttribute(&thr_sm, cudaDevAttrMaxThreadsPerMultiProcessor, dev) !=
          cudaSuccess ||
      cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) !=
          cudaSuccess)
    return 0;
  const size_t per_block = dyn_smem + fa.sharedSizeBytes + (size_t)reserved;
  const int warps = (threads + 31) / 32;
  const int regs_block = warps * (((fa.numRegs * 32) + 255) / 256) * 256;
  int n = thr_sm / threads;
  if (per_block > 0 && (int)((size_t)smem_sm / per_block) < n) n = (int)(smem_sm / per_block);
  if (regs_block > 0 && regs_sm / regs_block < n) n = regs_sm / regs_block;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&api, kern, threads, dyn_smem) ==
          cudaSuccess &&
      api > n)
    n = api;
  return n;
}

// Launch set-up of one (device, kernel, shared-memory size): the attributes
// are set once and the first wave's size (CTAs that fit at once on all SMs)
// is computed once; later launches reuse it without querying the driver.
struct VerifySetup {
  int dev;
  const void *kern;
  size_t smem;
  int first_wave;
};

cudaError_t verify_setup(const void *kern, int threads, size_t smem, int *first_wave) {
  static std::mutex mu;
  static VerifySetup cache[64];
  static int used = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  for (int k = 0; k < used; ++k)
    if (cache[k].dev == dev && cache[k].kern == kern && cache[k].smem == smem) {
      *first_wave = cache[k].first_wave;
      return cudaSuccess;
    }
  // the kernel's dynamic shared-memory limit is one attribute for every
  // launch of it: raise it to the device's opt-in maximum (never lower it to
  // this launch's size, which would break a cached larger configuration)
  // (the opt-in maximum less the kernel's static shared memory)
  int optin = 0;
  cudaFuncAttributes fa;
  cudaError_t e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  const int dyn_max = optin - (int)fa.sharedSizeBytes;
  if (dyn_max < 0 || (size_t)dyn_max < smem) return cudaErrorInvalidValue;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_max);
  if (e != cudaSuccess) return e;
  // all of the unified L1 as shared memory: two CTAs per SM at d = 128
  cudaError_t ce = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                        (int)cudaSharedmemCarveoutMaxShared);
  if (ce != cudaSuccess) return ce;
  const int per_sm = resident_ctas(kern, threads, smem);
  int sms = 0;
  *first_wave = per_sm > 0 && cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount,
                                                     dev) == cudaSuccess
                    ? per_sm * sms
                    : 0;
  if (used < 64) cache[used++] = VerifySetup{dev, kern, smem, *first_wave};
  return cudaSuccess;
}

template <int D, typename Tin>
cudaError_t launch_verify_t(VerifyParams p, cudaStream_t s) {
  const size_t smem = verify_smem_bytes(D, p.depth, p.max_T,
                                       sizeof(Tin) == 2 ? KDA_BF16 : KDA_F32);
  auto kern = p.max_T <= 8 ? verify_kernel<D, Tin, 8> : verify_kernel<D, Tin, 16>;
  // CTAs resident in the first wave: they prefetch the later waves' states.
  int first_wave = 0;
  cudaError_t e = verify_setup(reinterpret_cast<const void *>(kern), 2 * D, smem, &first_wave);
  if (e != cudaSuccess) return e;
  p.prefetch_stride = first_wave;
  // a programmatic dependent of the previous kernel on the stream: the
  // kernel prefetches into L2 before it waits for that kernel to complete
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.H, p.B);
  cfg.blockDim = dim3(2 * D);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace

size_t verify_smem_bytes(int D, int depth, int max_T, kda_dtype dt) {
#define KDA_S(DD)                                                            \
  case DD:                                                                   \
    return dt == KDA_BF16 ? Smem<DD, __nv_bfloat16>(depth, max_T).total      \
                          : Smem<DD, float>(depth, max_T).total;
  switch (D) {
    KDA_S(16)
    KDA_S(32)
    KDA_S(64)
    KDA_S(128)
    default:
      return 0;
  }
#undef KDA_S
}

int verify_max_spec_tokens() { return kTMax; }

cudaError_t launch_verify(const VerifyParams &p, kda_dtype dt, int D,
                          cudaStream_t s) {
  if (p.B == 0) return cudaSuccess;
  if (verify_pipe_applies(p, dt, D)) return launch_verify_pipe(p, s);
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

template <int D, typename Tin>
cudaError_t launch_verify_snapshot_t(const SnapshotParams &p, cudaStream_t s) {
  const size_t smem = (size_t)p.max_T * Rec<D, Tin>::kBytes;  // <= 33 KB
  verify_snapshot_kernel<D, Tin><<<dim3(p.H, p.B), 2 * D, smem, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_verify_snapshot(const SnapshotParams &p, kda_dtype dt, int D,
                                   cudaStream_t s) {
  if (p.B == 0) return cudaSuccess;
#define KDA_SV(DD)                                                          \
  case DD:                                                                  \
    return dt == KDA_BF16 ? launch_verify_snapshot_t<DD, __nv_bfloat16>(p, s) \
                          : launch_verify_snapshot_t<DD, float>(p, s);
  switch (D) {
    KDA_SV(16)
    KDA_SV(32)
    KDA_SV(64)
    KDA_SV(128)
    default:
      return cudaErrorInvalidValue;
  }
#undef KDA_SV
}

cudaError_t launch_commit_snapshot(const SnapshotParams &p, int D, cudaStream_t s) {
  if (p.B == 0) return cudaSuccess;
  const dim3 grid(p.H, p.B);
  switch (D) {
    case 16: commit_snapshot_kernel<16><<<grid, 256, 0, s>>>(p); break;
    case 32: commit_snapshot_kernel<32><<<grid, 256, 0, s>>>(p); break;
    case 64: commit_snapshot_kernel<64><<<grid, 256, 0, s>>>(p); break;
    case 128: commit_snapshot_kernel<128><<<grid, 256, 0, s>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace kda
