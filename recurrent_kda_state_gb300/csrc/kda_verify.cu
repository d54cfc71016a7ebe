// Verify + lazily fused ReplaySSM commit + ordinary decode, one kernel.
//
// One CTA owns one (sequence, head) unit for the whole launch, so the state of
// that unit is read from HBM once and written at most once:
//   1. replay the `accepted` ring entries recorded by the last commit onto the
//      state (token by token, kda_step), then write the committed state once;
//   2. speculative rows: evaluate the T drafted tokens from the committed
//      state in registers (outputs only, no draft state is stored) and copy
//      their inputs into the ring;  ordinary rows: apply the tokens and commit.
// ("ReplaySSM shrinks rollback state" and "Small tensor copies leave the hot
// path", vLLM Kimi K3 optimisation page.)
//
// Thread mapping for head dim D (d_k == d_v == D): 2*D threads; a thread owns
// value columns j0 = 2*(tid/4) and j0+1 of S and, of each, the key rows
// c = 4*(rg + 4*i) + {0..3}, i < D/16, rg = tid % 4.  The four threads of a
// column reduce with two xor-shuffles.  The state stays in registers.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr unsigned kFull = 0xffffffffu;

// Per-token record in shared memory (fp32): k[D] alpha[D] q[D] v[D] beta pad3.
template <int D>
struct Rec {
  static constexpr int kStride = 4 * D + 4;
  static constexpr int kK = 0, kA = D, kQ = 2 * D, kV = 3 * D, kB = 4 * D;
};

// One token of the recurrence on the thread's slice of S, fixed rounding:
//   S' = Diag(alpha) S;  dot_j = sum_c k_c S'_cj;  delta_j = beta (v_j - dot_j)
//   S  = S' + k delta^T;  o_j = sum_c q_c S_cj  (when WANT_O)
// This is the only place the committed state is advanced, so replay, decode
// and commit produce identical bits for identical inputs.
template <int D, bool WANT_O>
__device__ __forceinline__ void kda_step(float (&S)[2][D / 4], const float *rec,
                                         int rg, int j0, float &o0, float &o1) {
  constexpr int F = D / 16;
  const float4 *k4 = reinterpret_cast<const float4 *>(rec + Rec<D>::kK);
  const float4 *a4 = reinterpret_cast<const float4 *>(rec + Rec<D>::kA);
  const float4 *q4 = reinterpret_cast<const float4 *>(rec + Rec<D>::kQ);
  float d0 = 0.f, d1 = 0.f;
#pragma unroll
  for (int i = 0; i < F; ++i) {
    const float4 kk = k4[rg + 4 * i];
    const float4 aa = a4[rg + 4 * i];
    const float kv[4] = {kk.x, kk.y, kk.z, kk.w};
    const float av[4] = {aa.x, aa.y, aa.z, aa.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      S[0][4 * i + e] = __fmul_rn(S[0][4 * i + e], av[e]);
      d0 = __fmaf_rn(kv[e], S[0][4 * i + e], d0);
      S[1][4 * i + e] = __fmul_rn(S[1][4 * i + e], av[e]);
      d1 = __fmaf_rn(kv[e], S[1][4 * i + e], d1);
    }
  }
  d0 = __fadd_rn(d0, __shfl_xor_sync(kFull, d0, 1));
  d1 = __fadd_rn(d1, __shfl_xor_sync(kFull, d1, 1));
  d0 = __fadd_rn(d0, __shfl_xor_sync(kFull, d0, 2));
  d1 = __fadd_rn(d1, __shfl_xor_sync(kFull, d1, 2));
  const float beta = rec[Rec<D>::kB];
  const float del0 = __fmul_rn(beta, __fsub_rn(rec[Rec<D>::kV + j0], d0));
  const float del1 = __fmul_rn(beta, __fsub_rn(rec[Rec<D>::kV + j0 + 1], d1));
  float p0 = 0.f, p1 = 0.f;
#pragma unroll
  for (int i = 0; i < F; ++i) {
    const float4 kk = k4[rg + 4 * i];
    const float kv[4] = {kk.x, kk.y, kk.z, kk.w};
    float qv[4] = {0.f, 0.f, 0.f, 0.f};
    if (WANT_O) {
      const float4 qq = q4[rg + 4 * i];
      qv[0] = qq.x; qv[1] = qq.y; qv[2] = qq.z; qv[3] = qq.w;
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      S[0][4 * i + e] = __fmaf_rn(kv[e], del0, S[0][4 * i + e]);
      S[1][4 * i + e] = __fmaf_rn(kv[e], del1, S[1][4 * i + e]);
      if (WANT_O) {
        p0 = __fmaf_rn(qv[e], S[0][4 * i + e], p0);
        p1 = __fmaf_rn(qv[e], S[1][4 * i + e], p1);
      }
    }
  }
  if (WANT_O) {
    p0 += __shfl_xor_sync(kFull, p0, 1);
    p1 += __shfl_xor_sync(kFull, p1, 1);
    p0 += __shfl_xor_sync(kFull, p0, 2);
    p1 += __shfl_xor_sync(kFull, p1, 2);
    o0 = p0;
    o1 = p1;
  }
}

// Copy `count` token records into shared memory, converting to fp32.
// Source rows: element (t, h) of a packed [rows][H][D] tensor at row0 + t, or
// ring entries (base + t) of one (slot, head).
template <int D, typename Tin>
__device__ __forceinline__ void load_records(float *sm, int count,
                                             const Tin *k, const Tin *a,
                                             const Tin *q, const Tin *v,
                                             const Tin *b, size_t row_stride,
                                             size_t b_stride, int tid, int nt) {
  constexpr int E = InVec<Tin>::kElems;
  constexpr int CH = D / E;  // 16-byte chunks per vector
  const int nvec = q ? 4 : 3;
  const int total = count * nvec * CH;
  for (int idx = tid; idx < total; idx += nt) {
    const int t = idx / (nvec * CH);
    const int r = idx - t * nvec * CH;
    const int which = r / CH;
    const int ch = r - which * CH;
    const Tin *src = which == 0 ? k : which == 1 ? a : which == 2 ? v : q;
    const int off = which == 0 ? Rec<D>::kK : which == 1 ? Rec<D>::kA
                  : which == 2 ? Rec<D>::kV : Rec<D>::kQ;
    float tmp[E];
    InVec<Tin>::load(src + (size_t)t * row_stride + ch * E, tmp);
    float *dst = sm + t * Rec<D>::kStride + off + ch * E;
#pragma unroll
    for (int e = 0; e < E; e += 4)
      *reinterpret_cast<float4 *>(dst + e) =
          make_float4(tmp[e], tmp[e + 1], tmp[e + 2], tmp[e + 3]);
  }
  for (int t = tid; t < count; t += nt)
    sm[t * Rec<D>::kStride + Rec<D>::kB] = in_scalar<Tin>(b + (size_t)t * b_stride);
}

template <int D, typename Tin>
__global__ void __launch_bounds__(2 * D)
    verify_kernel(const VerifyParams p) {
  constexpr int NT = 2 * D;
  constexpr int R = D / 4;
  constexpr int F = D / 16;
  extern __shared__ float4 smem4[];
  float *sm = reinterpret_cast<float *>(smem4);
  __shared__ int s_info[6];  // skip, slot, accepted, T, tok0, spec

  const int h = blockIdx.x;
  const int i = blockIdx.y;
  const int tid = threadIdx.x;
  const int H = p.H;

  if (tid == 0) {
    int skip = 0, slot = p.state_slots[i], acc = 0, T = 0, tok0 = 0, spec = 0;
    if (slot < 0 || slot >= p.P) {
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
      const int32_t *c = p.ctrl + ((size_t)slot * H + h) * 2;
      const int pend = c[0];
      acc = c[1];
      if (pend < 0 || pend > p.depth || acc < 0 || acc > pend) {
        set_error(p.err, KDA_DERR_RING);
        skip = 1;
      }
    }
    s_info[0] = skip; s_info[1] = slot; s_info[2] = acc;
    s_info[3] = T; s_info[4] = tok0; s_info[5] = spec;
  }
  __syncthreads();
  if (s_info[0]) return;
  const int slot = s_info[1], acc = s_info[2], T = s_info[3];
  const int tok0 = s_info[4];
  const bool spec = s_info[5] != 0;

  const int rg = tid & 3;
  const int j0 = 2 * (tid >> 2);
  float *st = p.pool + ((size_t)slot * H + h) * D * D;

  // 1. state -> registers (128-bit loads; 4 lanes cover 64 contiguous bytes)
  float S[2][R];
  {
    const float4 *c0 = reinterpret_cast<const float4 *>(st + (size_t)j0 * D);
    const float4 *c1 = c0 + D / 4;
#pragma unroll
    for (int f = 0; f < F; ++f) {
      const float4 x = c0[rg + 4 * f];
      const float4 y = c1[rg + 4 * f];
      S[0][4 * f] = x.x; S[0][4 * f + 1] = x.y; S[0][4 * f + 2] = x.z; S[0][4 * f + 3] = x.w;
      S[1][4 * f] = y.x; S[1][4 * f + 1] = y.y; S[1][4 * f + 2] = y.z; S[1][4 * f + 3] = y.w;
    }
  }

  // 2. ring entries to replay, and this launch's tokens, -> shared memory
  const size_t unit = (size_t)slot * H + h;
  const Tin *rk = reinterpret_cast<const Tin *>(p.rk) + unit * p.depth * D;
  const Tin *ra = reinterpret_cast<const Tin *>(p.ra) + unit * p.depth * D;
  const Tin *rv = reinterpret_cast<const Tin *>(p.rv) + unit * p.depth * D;
  const Tin *rb = reinterpret_cast<const Tin *>(p.rb) + unit * p.depth;
  if (acc > 0)
    load_records<D, Tin>(sm, acc, rk, ra, nullptr, rv, rb, D, 1, tid, NT);
  float *tsm = sm + p.depth * Rec<D>::kStride;
  if (T > 0) {
    const size_t row = (size_t)tok0 * H + h;
    load_records<D, Tin>(tsm, T,
                         reinterpret_cast<const Tin *>(p.k) + row * D,
                         reinterpret_cast<const Tin *>(p.alpha) + row * D,
                         reinterpret_cast<const Tin *>(p.q) + row * D,
                         reinterpret_cast<const Tin *>(p.v) + row * D,
                         reinterpret_cast<const Tin *>(p.beta) + row,
                         (size_t)H * D, (size_t)H, tid, NT);
  }
  __syncthreads();

  // 3. lazy commit: replay the accepted entries
  float o0 = 0.f, o1 = 0.f;
  for (int t = 0; t < acc; ++t)
    kda_step<D, false>(S, sm + t * Rec<D>::kStride, rg, j0, o0, o1);

  auto store_state = [&]() {
    float4 *c0 = reinterpret_cast<float4 *>(st + (size_t)j0 * D);
    float4 *c1 = c0 + D / 4;
#pragma unroll
    for (int f = 0; f < F; ++f) {
      c0[rg + 4 * f] = make_float4(S[0][4 * f], S[0][4 * f + 1], S[0][4 * f + 2], S[0][4 * f + 3]);
      c1[rg + 4 * f] = make_float4(S[1][4 * f], S[1][4 * f + 1], S[1][4 * f + 2], S[1][4 * f + 3]);
    }
  };

  if (spec) {
    if (acc > 0) store_state();
    // ring <- this launch's drafted inputs (old entries are already in smem)
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
    // drafts: outputs from the committed state; the draft states die here
    for (int t = 0; t < T; ++t) {
      kda_step<D, true>(S, tsm + t * Rec<D>::kStride, rg, j0, o0, o1);
      if (rg == 0)
        *reinterpret_cast<float2 *>(p.o + ((size_t)(tok0 + t) * H + h) * D + j0) =
            make_float2(o0, o1);
    }
    if (tid == 0) {
      int32_t *c = p.ctrl + unit * 2;
      c[0] = T;
      c[1] = 0;
    }
  } else {
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
cudaError_t launch_verify_t(const VerifyParams &p, cudaStream_t s) {
  const size_t smem = (size_t)(p.depth + p.max_T) * Rec<D>::kStride * sizeof(float);
  auto kern = verify_kernel<D, Tin>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(
        kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  dim3 grid(p.H, p.B);
  kern<<<grid, 2 * D, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

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

cudaError_t launch_ring_reset(const CommitParams &p, cudaStream_t s) {
  const int n = p.B * p.H;
  if (n == 0) return cudaSuccess;
  ring_reset_kernel<<<(n + 255) / 256, 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace kda
