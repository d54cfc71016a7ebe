// Chunked prefill with in-pass state checkpoints.
// ("KDA checkpoints stay inside the prefill", vLLM Kimi K3 optimisation page:
// the checkpoint at a cache-block boundary is exported by the same pass.)
//
// Chunk-wise (WY/UT) form of the gated delta rule, per chunk of C tokens
// aligned to absolute positions, g_t = sum_{s<=t} log alpha_s per key channel:
//   A    = strict_tril(diag(beta) (e^{g} K)(e^{-g} K)^T),  T = (I + A)^{-1} diag(beta)
//   W    = T (e^{g} K),  U' = T V,  U = U' - W S
//   O    = (e^{g} Q) S + tril(( e^{g} Q)(e^{-g} K)^T) U
//   S'   = Diag(e^{g_C}) S + (e^{g_C - g} K)^T U
// The e^{g} / e^{-g} pair inside A and M is referenced to the chunk's middle
// row so both factors stay near 1; every other factor is <= 1.
//
// Three launches:
//   chunk_table   one thread: per-sequence chunk offsets into the workspace;
//   intra         grid (chunk, head): everything that does not depend on S
//                 (W, U', e^{g}Q, e^{g_C-g}K, M, e^{g_C}) -> workspace;
//   state         grid (value-column slice, head, sequence): the sequential
//                 pass over chunks; U, O, S' per chunk; checkpoints.
#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int kNT = 256;

// Entry layout (floats): W [C][D], U' [C][D], Qg [C][D], Kb [C][D], M [C][C], gC [D]
template <int D, int C>
struct Entry {
  static constexpr int kW = 0, kU = C * D, kQ = 2 * C * D, kKb = 3 * C * D;
  static constexpr int kM = 4 * C * D, kG = 4 * C * D + C * C;
};

__global__ void chunk_table_kernel(const PrefillParams p, int C) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  int *table = reinterpret_cast<int *>(p.ws);
  int off = 0;
  for (int i = 0; i < p.B; ++i) {
    table[i] = off;
    const int c0 = p.cu_seqlens[i], c1 = p.cu_seqlens[i + 1];
    int L = c1 - c0;
    if (c0 < 0 || L < 0 || c1 > p.N) {
      set_error(p.err, KDA_DERR_SEGMENT);
      L = 0;
    }
    int p0 = p.start_pos ? p.start_pos[i] : 0;
    if (p0 < 0) {
      set_error(p.err, KDA_DERR_SEGMENT);
      L = 0;
      p0 = 0;
    }
    const int r = p0 % C;
    int nch = L > 0 ? (r + L + C - 1) / C : 0;
    if (off + nch > p.max_chunks) {
      set_error(p.err, KDA_DERR_SEGMENT);
      nch = 0;
    }
    off += nch;
  }
  table[p.B] = off;
}

// Load rows t < n of one input vector (head h) as fp32 into dst[t * ld + c];
// rows n..C-1 are filled with `pad`.  Optional elementwise transform.
template <int D, int C, typename Tin, typename F>
__device__ __forceinline__ void load_rows(float *dst, int ld, const Tin *src,
                                          int tok0, int n, int H, int h,
                                          float pad, int tid, F f) {
  constexpr int E = InVec<Tin>::kElems;
  constexpr int CH = D / E;
  for (int idx = tid; idx < C * CH; idx += kNT) {
    const int t = idx / CH, ch = idx - (idx / CH) * CH;
    float tmp[E];
    if (t < n) {
      InVec<Tin>::load(src + ((size_t)(tok0 + t) * H + h) * D + ch * E, tmp);
#pragma unroll
      for (int e = 0; e < E; ++e) tmp[e] = f(tmp[e], t, ch * E + e);
    } else {
#pragma unroll
      for (int e = 0; e < E; ++e) tmp[e] = pad;
    }
#pragma unroll
    for (int e = 0; e < E; e += 4)
      *reinterpret_cast<float4 *>(dst + t * ld + ch * E + e) =
          make_float4(tmp[e], tmp[e + 1], tmp[e + 2], tmp[e + 3]);
  }
}

// out[t][s] = mask(t, s) * scale(t) * dot(Xr[t], Yr[s]) over D, t, s < C.
// 4x4 register tiles with interleaved rows (t = tb + C/4 * a) so that the
// 16-byte shared loads of one warp phase fall in distinct banks.
template <int D, int C, bool STRICT>
__device__ __forceinline__ void gram_tril(float *out, int ldo, const float *Xr,
                                          const float *Yr, int ld,
                                          const float *scale, int tid) {
  constexpr int N4 = C / 4;
  for (int tile = tid; tile < N4 * N4; tile += kNT) {
    const int tb = tile / N4, sb = tile - (tile / N4) * N4;
    float acc[4][4] = {};
    for (int c = 0; c < D; c += 4) {
      float4 x[4], y[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        x[a] = *reinterpret_cast<const float4 *>(Xr + (tb + N4 * a) * ld + c);
        y[a] = *reinterpret_cast<const float4 *>(Yr + (sb + N4 * a) * ld + c);
      }
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          acc[a][b] = fmaf(x[a].x, y[b].x, acc[a][b]);
          acc[a][b] = fmaf(x[a].y, y[b].y, acc[a][b]);
          acc[a][b] = fmaf(x[a].z, y[b].z, acc[a][b]);
          acc[a][b] = fmaf(x[a].w, y[b].w, acc[a][b]);
        }
    }
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int t = tb + N4 * a, s = sb + N4 * b;
        const bool keep = STRICT ? (s < t) : (s <= t);
        out[t * ldo + s] = keep ? (scale ? scale[t] : 1.f) * acc[a][b] : 0.f;
      }
  }
}

// dst[t][c] (global, row stride D) = sum_s Tm[t][s] Y[s][c], t < C, c < D.
template <int D, int C>
__device__ __forceinline__ void tri_apply(float *dst, const float *Tm, int ldt,
                                          const float *Y, int ld, int tid) {
  constexpr int N4 = C / 4, D4 = D / 4;
  for (int tile = tid; tile < N4 * D4; tile += kNT) {
    const int tb = tile / D4, cc = tile - (tile / D4) * D4;
    float4 acc[4];
#pragma unroll
    for (int a = 0; a < 4; ++a) acc[a] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < C; ++s) {
      const float4 y = *reinterpret_cast<const float4 *>(Y + s * ld + 4 * cc);
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const float tv = Tm[(tb + N4 * a) * ldt + s];
        acc[a].x = fmaf(tv, y.x, acc[a].x);
        acc[a].y = fmaf(tv, y.y, acc[a].y);
        acc[a].z = fmaf(tv, y.z, acc[a].z);
        acc[a].w = fmaf(tv, y.w, acc[a].w);
      }
    }
#pragma unroll
    for (int a = 0; a < 4; ++a)
      *reinterpret_cast<float4 *>(dst + (size_t)(tb + N4 * a) * D + 4 * cc) = acc[a];
  }
}

template <int D, int C, typename Tin>
__global__ void __launch_bounds__(kNT) prefill_intra_kernel(const PrefillParams p) {
  constexpr int LD = D + 4, LC = C + 4;
  extern __shared__ float4 smem4[];
  float *Kr = reinterpret_cast<float *>(smem4);
  float *G = Kr + C * LD;
  float *X = G + C * LD;
  float *Y = X + C * LD;
  float *A = Y + C * LD;
  float *Tm = A + C * LC;
  float *Mq = Tm + C * LC;
  float *bet = Mq + C * LC;
  float *gm = bet + C;

  const int g = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  const int total = reinterpret_cast<const int *>(p.ws)[p.B];
  if (g >= total) return;
  const ChunkLoc cl = locate_chunk(p, g, C);
  const int n = cl.n, tok0 = cl.tok0, H = p.H;
  float *ent = reinterpret_cast<float *>(p.ws + prefill_table_bytes(p.B)) +
               ((size_t)g * H + h) * prefill_entry_floats(D, C);

  const Tin *qin = reinterpret_cast<const Tin *>(p.q);
  const Tin *kin = reinterpret_cast<const Tin *>(p.k);
  const Tin *vin = reinterpret_cast<const Tin *>(p.v);
  const Tin *ain = reinterpret_cast<const Tin *>(p.alpha);
  const Tin *bin = reinterpret_cast<const Tin *>(p.beta);
  auto ident = [] __device__(float x, int, int) { return x; };

  // 1. raw k, log alpha (padded rows: k = 0, log alpha = 0), beta
  load_rows<D, C, Tin>(Kr, LD, kin, tok0, n, H, h, 0.f, tid, ident);
  load_rows<D, C, Tin>(G, LD, ain, tok0, n, H, h, 0.f, tid,
                       [] __device__(float x, int, int) { return logf(x); });
  for (int t = tid; t < C; t += kNT)
    bet[t] = t < n ? in_scalar<Tin>(bin + (size_t)(tok0 + t) * H + h) : 0.f;
  __syncthreads();
  // 2. inclusive cumulative log-decay per key channel
  for (int c = tid; c < D; c += kNT) {
    float acc = 0.f;
    for (int t = 0; t < C; ++t) {
      acc += G[t * LD + c];
      G[t * LD + c] = acc;
    }
  }
  __syncthreads();
  // 3. factors referenced to the middle row m
  const int m = n / 2;
  for (int c = tid; c < D; c += kNT) {
    gm[c] = G[m * LD + c];
    if (G[c] - G[m * LD + c] > 80.f || G[m * LD + c] - G[(C - 1) * LD + c] > 80.f)
      set_error(p.err, KDA_DERR_RANGE);
  }
  __syncthreads();
  for (int idx = tid; idx < C * D; idx += kNT) {
    const int t = idx / D, c = idx - (idx / D) * D;
    const float dg = G[t * LD + c] - gm[c];
    X[t * LD + c] = expf(dg) * Kr[t * LD + c];
    Y[t * LD + c] = expf(-dg) * Kr[t * LD + c];
  }
  __syncthreads();
  // 4. A = strict_tril(diag(beta) X Y^T)
  gram_tril<D, C, true>(A, LC, X, Y, LD, bet, tid);
  __syncthreads();
  // 5. Z = e^{g - g_m} q into X; M = tril(Z Y^T)
  load_rows<D, C, Tin>(X, LD, qin, tok0, n, H, h, 0.f, tid,
                       [=] __device__(float x, int t, int c) {
                         return expf(G[t * LD + c] - gm[c]) * x;
                       });
  __syncthreads();
  gram_tril<D, C, false>(Mq, LC, X, Y, LD, nullptr, tid);
  __syncthreads();
  // 6. T = (I + A)^{-1} diag(beta): one column per thread, forward substitution
  if (tid < C) {
    const int s = tid;
    float Tc[C];
#pragma unroll
    for (int t = 0; t < C; ++t) {
      float acc = 0.f;
#pragma unroll
      for (int r = 0; r < t; ++r) acc = fmaf(A[t * LC + r], Tc[r], acc);
      Tc[t] = t < s ? 0.f : (t == s ? bet[t] : -acc);
    }
#pragma unroll
    for (int t = 0; t < C; ++t) Tm[t * LC + s] = Tc[t];
  }
  // K~ = e^{g} k into Y (Y no longer read once M is done)
  for (int idx = tid; idx < C * D; idx += kNT) {
    const int t = idx / D, c = idx - (idx / D) * D;
    Y[t * LD + c] = expf(G[t * LD + c]) * Kr[t * LD + c];
  }
  __syncthreads();
  // 7. W = T K~ ; then V into X and U' = T V
  tri_apply<D, C>(ent + Entry<D, C>::kW, Tm, LC, Y, LD, tid);
  load_rows<D, C, Tin>(X, LD, vin, tok0, n, H, h, 0.f, tid, ident);
  __syncthreads();
  tri_apply<D, C>(ent + Entry<D, C>::kU, Tm, LC, X, LD, tid);
  // 8. e^{g} q, e^{g_C - g} k, M, e^{g_C} -> workspace
  {
    constexpr int E = InVec<Tin>::kElems;
    constexpr int CH = D / E;
    for (int idx = tid; idx < C * CH; idx += kNT) {
      const int t = idx / CH, ch = idx - (idx / CH) * CH;
      float tmp[E];
      if (t < n)
        InVec<Tin>::load(qin + ((size_t)(tok0 + t) * H + h) * D + ch * E, tmp);
      else
        for (int e = 0; e < E; ++e) tmp[e] = 0.f;
      float *dq = ent + Entry<D, C>::kQ + t * D + ch * E;
      float *dk = ent + Entry<D, C>::kKb + t * D + ch * E;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const int c = ch * E + e;
        dq[e] = expf(G[t * LD + c]) * tmp[e];
        dk[e] = expf(G[(C - 1) * LD + c] - G[t * LD + c]) * Kr[t * LD + c];
      }
    }
    for (int idx = tid; idx < C * C; idx += kNT) {
      const int t = idx / C, s = idx - (idx / C) * C;
      ent[Entry<D, C>::kM + idx] = Mq[t * LC + s];
    }
    for (int c = tid; c < D; c += kNT)
      ent[Entry<D, C>::kG + c] = expf(G[(C - 1) * LD + c]);
  }
}

template <int D, int C>
__global__ void __launch_bounds__(kNT) prefill_state_kernel(const PrefillParams p) {
  constexpr int NC = D < 32 ? D : 32;  // value columns per CTA
  constexpr int LD = D + 4, LC = C + 4, LS = NC + 1;
  constexpr int GR = kNT / NC;         // thread groups sharing a column
  constexpr int RPT = C / GR;          // token rows per thread
  constexpr int CPT = D / GR;          // key rows per thread (state update)
  static_assert(RPT >= 1 && CPT >= 1 && GR * NC == kNT, "tile shape");
  extern __shared__ float4 smem4[];
  float *Ss = reinterpret_cast<float *>(smem4);  // [D][LS]
  float *W = Ss + D * LS;                         // [C][LD]
  float *Qg = W + C * LD;
  float *Kb = Qg + C * LD;
  float *M = Kb + C * LD;                         // [C][LC]
  float *Up = M + C * LC;                         // [C][NC]
  float *U = Up + C * NC;                         // [C][NC]
  float *gC = U + C * NC;                         // [D]

  const int sl = blockIdx.x, h = blockIdx.y, i = blockIdx.z, tid = threadIdx.x;
  const int H = p.H, col0 = sl * NC;
  const int *table = reinterpret_cast<const int *>(p.ws);
  const int g0 = table[i], nch = table[i + 1] - table[i];
  if (nch <= 0) return;
  const int slot = p.state_slots[i];
  if (slot < 0 || slot >= p.P) {
    if (tid == 0 && sl == 0) set_error(p.err, KDA_DERR_SLOT);
    return;
  }
  const float *wsf = reinterpret_cast<const float *>(p.ws + prefill_table_bytes(p.B));
  const int cu0 = p.cu_seqlens[i];
  const int L = p.cu_seqlens[i + 1] - cu0;
  const int p0 = p.start_pos ? p.start_pos[i] : 0;
  const int r0 = p0 % C;

  auto state_ptr = [&](int s) {
    return p.pool + (((size_t)s * H + h) * D + col0) * D;
  };
  {  // S slice -> smem, Ss[c][j] = S_{c, col0 + j}
    const float *src = state_ptr(slot);
    for (int idx = tid; idx < NC * D; idx += kNT) {
      const int j = idx / D, c = idx - (idx / D) * D;
      Ss[c * LS + j] = src[(size_t)j * D + c];
    }
  }
  const int j = tid % NC, grp = tid / NC;
  for (int q = 0; q < nch; ++q) {
    const float *ent = wsf + ((size_t)(g0 + q) * H + h) * prefill_entry_floats(D, C);
    for (int idx = tid; idx < C * (D / 4); idx += kNT) {
      const int t = idx / (D / 4), c4 = idx - (idx / (D / 4)) * (D / 4);
      *reinterpret_cast<float4 *>(W + t * LD + 4 * c4) =
          *reinterpret_cast<const float4 *>(ent + Entry<D, C>::kW + t * D + 4 * c4);
      *reinterpret_cast<float4 *>(Qg + t * LD + 4 * c4) =
          *reinterpret_cast<const float4 *>(ent + Entry<D, C>::kQ + t * D + 4 * c4);
      *reinterpret_cast<float4 *>(Kb + t * LD + 4 * c4) =
          *reinterpret_cast<const float4 *>(ent + Entry<D, C>::kKb + t * D + 4 * c4);
    }
    for (int idx = tid; idx < C * C; idx += kNT) {
      const int t = idx / C, s = idx - (idx / C) * C;
      M[t * LC + s] = ent[Entry<D, C>::kM + idx];
    }
    for (int idx = tid; idx < C * NC; idx += kNT) {
      const int t = idx / NC, jj = idx - (idx / NC) * NC;
      Up[idx] = ent[Entry<D, C>::kU + t * D + col0 + jj];
    }
    for (int c = tid; c < D; c += kNT) gC[c] = ent[Entry<D, C>::kG + c];
    __syncthreads();

    // U = U' - W S and R = Qg S for rows t = grp + GR * a
    float R[RPT];
    {
      float P[RPT];
#pragma unroll
      for (int a = 0; a < RPT; ++a) P[a] = R[a] = 0.f;
      for (int c = 0; c < D; c += 4) {
        const float s0 = Ss[c * LS + j], s1 = Ss[(c + 1) * LS + j];
        const float s2 = Ss[(c + 2) * LS + j], s3 = Ss[(c + 3) * LS + j];
#pragma unroll
        for (int a = 0; a < RPT; ++a) {
          const int t = grp + GR * a;
          const float4 w = *reinterpret_cast<const float4 *>(W + t * LD + c);
          const float4 x = *reinterpret_cast<const float4 *>(Qg + t * LD + c);
          P[a] = fmaf(w.x, s0, fmaf(w.y, s1, fmaf(w.z, s2, fmaf(w.w, s3, P[a]))));
          R[a] = fmaf(x.x, s0, fmaf(x.y, s1, fmaf(x.z, s2, fmaf(x.w, s3, R[a]))));
        }
      }
#pragma unroll
      for (int a = 0; a < RPT; ++a) {
        const int t = grp + GR * a;
        U[t * NC + j] = Up[t * NC + j] - P[a];
      }
    }
    __syncthreads();
    // O = Qg S + M U  (rows of this chunk that exist)
    const int s_loc = max(0, q * C - r0);
    const int e_loc = min(L, (q + 1) * C - r0);
    const int n = e_loc - s_loc;
#pragma unroll
    for (int a = 0; a < RPT; ++a) {
      const int t = grp + GR * a;
      float acc = R[a];
      for (int s = 0; s <= t; ++s) acc = fmaf(M[t * LC + s], U[s * NC + j], acc);
      if (t < n)
        p.o[((size_t)(cu0 + s_loc + t) * H + h) * D + col0 + j] = acc;
    }
    // S' = Diag(gC) S + Kb^T U for key rows c = grp * CPT + b
    {
      float acc[CPT];
#pragma unroll
      for (int b = 0; b < CPT; ++b) {
        const int c = grp * CPT + b;
        acc[b] = gC[c] * Ss[c * LS + j];
      }
      for (int t = 0; t < C; ++t) {
        const float u = U[t * NC + j];
        if constexpr (CPT % 4 == 0) {
#pragma unroll
          for (int b = 0; b < CPT; b += 4) {
            const float4 kb = *reinterpret_cast<const float4 *>(Kb + t * LD + grp * CPT + b);
            acc[b] = fmaf(kb.x, u, acc[b]);
            acc[b + 1] = fmaf(kb.y, u, acc[b + 1]);
            acc[b + 2] = fmaf(kb.z, u, acc[b + 2]);
            acc[b + 3] = fmaf(kb.w, u, acc[b + 3]);
          }
        } else {
#pragma unroll
          for (int b = 0; b < CPT; ++b)
            acc[b] = fmaf(Kb[t * LD + grp * CPT + b], u, acc[b]);
        }
      }
#pragma unroll
      for (int b = 0; b < CPT; ++b) Ss[(grp * CPT + b) * LS + j] = acc[b];
    }
    __syncthreads();
    // in-pass checkpoint at an absolute block boundary
    const int P_end = p0 + e_loc;
    if (p.ckpt_every > 0 && P_end % p.ckpt_every == 0 && p.ckpt_slots) {
      const int mth = P_end / p.ckpt_every - p0 / p.ckpt_every - 1;
      if (mth >= 0 && mth < p.max_ckpt) {
        const int cs = p.ckpt_slots[(size_t)i * p.max_ckpt + mth];
        if (cs >= p.P) {
          if (tid == 0 && sl == 0) set_error(p.err, KDA_DERR_SLOT);
        } else if (cs >= 0) {
          float *dst = state_ptr(cs);
          for (int idx = tid; idx < NC * D; idx += kNT) {
            const int jj = idx / D, c = idx - (idx / D) * D;
            dst[(size_t)jj * D + c] = Ss[c * LS + jj];
          }
        }
      }
    }
  }
  {
    float *dst = state_ptr(slot);
    for (int idx = tid; idx < NC * D; idx += kNT) {
      const int jj = idx / D, c = idx - (idx / D) * D;
      dst[(size_t)jj * D + c] = Ss[c * LS + jj];
    }
  }
}

template <int D, int C, typename Tin>
cudaError_t launch_prefill_t(const PrefillParams &p, cudaStream_t s) {
  constexpr int LD = D + 4, LC = C + 4;
  constexpr int NC = D < 32 ? D : 32;
  chunk_table_kernel<<<1, 32, 0, s>>>(p, C);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const size_t sm1 = (size_t)(4 * C * LD + 3 * C * LC + C + D) * sizeof(float);
  auto k1 = prefill_intra_kernel<D, C, Tin>;
  e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm1);
  if (e != cudaSuccess) return e;
  if (p.max_chunks > 0) {
    k1<<<dim3(p.max_chunks, p.H), kNT, sm1, s>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const size_t sm2 =
      (size_t)(D * (NC + 1) + 3 * C * LD + C * LC + 2 * C * NC + D) * sizeof(float);
  auto k2 = prefill_state_kernel<D, C>;
  e = cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm2);
  if (e != cudaSuccess) return e;
  k2<<<dim3(D / NC, p.H, p.B), kNT, sm2, s>>>(p);
  return cudaGetLastError();
}

template <int D, typename Tin>
cudaError_t launch_prefill_c(const PrefillParams &p, int C, cudaStream_t s) {
  switch (C) {
    case 16: return launch_prefill_t<D, 16, Tin>(p, s);
    case 32: return launch_prefill_t<D, 32, Tin>(p, s);
    case 64: return launch_prefill_t<D, 64, Tin>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_chunk_table(const PrefillParams &p, int C, cudaStream_t s) {
  chunk_table_kernel<<<1, 32, 0, s>>>(p, C);
  return cudaGetLastError();
}

cudaError_t launch_prefill(const PrefillParams &p, kda_dtype dt, int D, int C,
                           cudaStream_t s) {
  if (p.B == 0) return cudaSuccess;
  if (prefill_uses_tc(dt, p.H, D, D, C)) return launch_prefill_tc(p, s);
#define KDA_P(DD)                                                            \
  case DD:                                                                   \
    return dt == KDA_BF16 ? launch_prefill_c<DD, __nv_bfloat16>(p, C, s)     \
                          : launch_prefill_c<DD, float>(p, C, s);
  switch (D) {
    KDA_P(16)
    KDA_P(32)
    KDA_P(64)
    KDA_P(128)
    default:
      return cudaErrorInvalidValue;
  }
#undef KDA_P
}

}  // namespace kda
