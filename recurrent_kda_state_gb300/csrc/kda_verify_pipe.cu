// Verify + lazily fused ReplaySSM commit + ordinary decode as a persistent,
// warp-specialised pipeline: d_k = d_v = 128, bf16 inputs, ring depth <= 8,
// at most 8 tokens per row.  ("ReplaySSM shrinks rollback state" and "Small
// tensor copies leave the hot path", vLLM Kimi K3 optimisation page.)
//
// Each (sequence, head) unit computes exactly what verify_kernel computes --
// replay the accepted ring entries with kda_step, store the state once, then
// the drafted tokens' outputs from the committed state in chunk form, or the
// ordinary rows' tokens applied and committed -- and its state is read from
// HBM once and written at most once.  What changes is how the units flow
// through an SM: one CTA per SM walks the units u = blockIdx.x + n * gridDim.x
// with three roles working on different units at once:
//
//   producer (1 warp): the units' slot, segment, ring word and beta values
//       for 32 units at a time (one unit per lane); then per unit its 64 KiB
//       state as one 128-byte-swizzled TMA box (four 16 KB blocks of 32 key
//       channels) through a 3-D tensor map of the pool into one of two state
//       stages (two units ahead of the consumers), its token rows as four
//       TMA boxes (k, alpha, q, v: 8 tokens x 128 channels) and its pending
//       ring entries as three TMA boxes into one of three token stages, each
//       as soon as its stage is free (the first unit's rows as soon as its
//       segment is known), and an L2 hint for the next unit's state;
//   prep (groups of 2 warps taking units in turn: one group on prepared
//       inputs, two on projection-space inputs, see PipeRoles): as soon as a
//       unit's token stage lands, for drafts: the
//       decay products gamma_t, K~ = gamma k, Q~ = gamma q, K^ = k / gamma,
//       the T x T pair products A = K^ K~^T, B = K^ Q~^T on the tensor cores,
//       N = B (I + diag(beta) A)^-1 diag(beta) by back substitution, then
//       Q^ = Q~ - N K~ (as bf16 hi/lo MMA fragments) and W = N v, and the
//       unit's control word;
//   ring append (1 warp): after each unit's hand-off, its drafted inputs
//       into the unit's ring, outside the prep warps' barriers;
//   consumers (8 warps): the state from its stage into registers (the stage
//       is released at once), the replay as soon as the token stage lands
//       (while the prep still works on it), the state store, and once the
//       prep is done the drafts' outputs o_t = (S^T Q^)_t + W_t with bf16
//       hi/lo tensor-core MMAs taken straight from the registers that hold S.
//
// so that while the consumers work on one unit the next units' bytes are in
// flight: the kernel keeps HBM busy instead of alternating load and compute
// phases.  Every wait is bounded and per warp; a wait that runs out sets
// KDA_DERR_TIMEOUT, every role stops taking units, and the producer waits
// (bounded) for its copies in flight before the CTA exits.
//
// The consumers' thread mapping and kda_step are those of verify_kernel, so
// replayed states are bit-identical to ordinary decode in either kernel.
//
// Chunk form of the drafts.  With x_t = (S^T K~_t)_j and y_t = (S^T Q~_t)_j
// for value column j, the corrections delta = M (v_j - x) and the outputs
// o_t = y_t + sum_{s<=t} B_ts delta_s unroll the recurrence over the drafted
// tokens; substituting delta, o = S^T (Q~ - N K~) + N v_j with N = B M, so
// the consumers need one product S^T Q^ per unit and no solve.
//
// MMA mapping (mma.sync m16n8k16, bf16 in, fp32 accumulate).  Warp w owns the
// value columns 16w .. 16w+15; lane (g = lane/4, r = lane%4) holds columns
// j0 = 16w + 2g, j0 + 1 and key rows c = 16f + 4r + {0..3} of k-tile f.
// Reading A row g as column j0, row g + 8 as column j0 + 1, and the k index
// 2r + {0,1} as c = 16f + 4r + {0,1}, 2r + 8 + {0,1} as c = 16f + 4r + {2,3},
// the four state pairs of k-tile f are exactly the A fragment of that tile;
// B column n = drafted row t needs X[t][16f + 4r .. +3], which the prep warps
// store in fragment order.  D row g / g+8, column 2r + {0,1} is then
// (S^T X)_{j0 / j0+1, t = 2r + {0,1}}.  The pair products use K^ as A (rows
// s = 0..7, rows 8..15 zero) in the same k order, so D row s, column t is
// K^_s . X_t.
#include <cuda.h>

#include <cstddef>
#include <cstring>
#include <mutex>

#include "kda_internal.cuh"
#include "kda_step.cuh"
#include "kda_umma.cuh"

namespace kda {
namespace {

constexpr int PD = 128;                 // head dim
constexpr int PT = 8;                   // drafted rows per MMA tile (T <= 8)
constexpr int kDepthMax = 8;            // ring entries a stage holds
constexpr int kConsumerWarps = 8;       // 2 * PD threads: the state owners
constexpr int kProducerWarp = 8;
// Prep groups of two channel-pair warps take units in turn; one more warp
// appends to the ring.  On prepared inputs one group (twelve warps, three
// per scheduler, so the consumers keep the registers they use); on
// projection-space inputs, whose prep also normalises keys and maps the
// decay and beta logits, two groups prepare two units at once (fourteen
// warps put four on two schedulers, whose 16 K registers then cap every
// thread at 128: slower consumers, paid for by the heavier prep's overlap).
constexpr int kPrepWarp0 = 9;
constexpr int kPrepMath = 64;           // a group's two channel-pair warps
template <bool RAW>
struct PipeRoles {
  static constexpr int kGroups = RAW ? 2 : 1;
  static constexpr int kRingWarp = kPrepWarp0 + 2 * kGroups;
  static constexpr int kPrepWarps = 2 * kGroups + 1;  // with the ring warp
  static constexpr int kThreads = 32 * (kConsumerWarps + 1 + kPrepWarps);
};
// named barriers of group g: kPrepBar + 2 g (its 64 threads), kPrepChanBar + 2 g
constexpr int kPrepBar = 1;
constexpr int kPrepChanBar = 2;
constexpr int kTStages = 3;             // token stages
constexpr int kSStages = 2;             // state stages
constexpr int kMetaBatch = 32;          // units whose words one lane each reads at once
constexpr int kMetaRing = 2 * kMetaBatch;

typedef __nv_bfloat16 bf16;
// A token stage's rows: dense [PT][PD] arrays of k, alpha, q and v (row t =
// token t: the layout one TMA box of PT tokens x PD channels lands in), then
// beta [PT].  Channel c of token t's field X is at X + t * kStride + c; the
// beta of token t at kB + t.
struct R {
  static constexpr int kStride = PD;
  static constexpr int kK = 0, kA = PT * PD, kQ = 2 * PT * PD, kV = 3 * PT * PD;
  static constexpr int kB = 4 * PT * PD;
  static constexpr int kBytes = (kB + PT) * 2;
};

// The packed token tensors [N][H][PD] (bf16) as 3-D tensor maps with boxes of
// PD channels x 1 head x PT tokens (rows past N read as zeros).
struct TokMaps {
  CUtensorMap k, a, q, v;
  CUtensorMap rk, ra, rv;  // the ring payload [P * H][depth][PD], boxes of depth entries
  int tok_rows, ring_rows;  // box heights: min(PT, N) tokens, depth (<= 8) entries
};
static_assert(offsetof(TokMaps, rv) == offsetof(TokMaps, k) + 6 * sizeof(CUtensorMap),
              "the seven maps are consecutive");

// Per-unit facts the producer hands to the other roles.
struct UnitMeta {
  int slot, tok0, T, spec, acc, skip, pad0, pad1;
};
// The producer's copy of a unit's words: the meta and the beta values it
// places (ring entries 0..7, then drafted tokens 0..7), raw input bits.
struct MetaEnt {
  UnitMeta m;
  unsigned short b[16];
};
static_assert(sizeof(MetaEnt) == 64, "meta ring entries are 64 bytes");

// Shared-memory carve-up, byte offsets from a 1024-aligned base.
struct PipeLayout {
  // state stage: state [PD][PD] fp32 as four 16 KB blocks of 32 key channels
  // x 128 value rows (row j = value column, 128 bytes, its 16-byte chunks
  // swizzled by j % 8: the TMA 128-byte swizzle), then the meta (slot and
  // whether the state was loaded); stages 1024-byte aligned for the swizzle
  static constexpr int kSsState = 0;
  static constexpr int kSsMeta = PD * PD * 4;
  static constexpr int kSStage = (kSsMeta + (int)sizeof(UnitMeta) + 1023) & ~1023;
  // token stage:
  //   rec   the drafted / ordinary tokens (R layout, input dtype)
  //   rv    pending ring entries' v [8][PD] (input dtype), rb their beta [8]
  //   rk    pending ring entries' k, alpha [2][8][PD] (input dtype)
  //   frag  three regions of 8 k-tiles x 32 lanes x {hi01, hi23, lo01, lo23}:
  //         the MMA fragments of K~, Q~ (then Q^), K^ (then W, fp32 [PT][PD])
  //   am bm pair matrices A, B [PT][PT] fp32; flag (explicit pair products);
  //   n     N = B M [PT][PT] fp32; meta (complete).  Once the pair
  //         products are taken, the K~ fragments' region holds the small
  //         matrices that give M.
  // (the TMA boxes' destinations -- the four token fields, rv and both
  // halves of rk -- start on 128-byte boundaries)
  static constexpr int kTsRec = 0;
  static constexpr int kTsRv = (kTsRec + R::kBytes + 127) & ~127;
  static constexpr int kTsRb = kTsRv + kDepthMax * PD * 2;
  static constexpr int kTsRk = (kTsRb + 16 + 127) & ~127;
  static constexpr int kTsFrag = kTsRk + 2 * kDepthMax * PD * 2;
  static constexpr int kTsAm = kTsFrag + 3 * 8 * 32 * 16;
  static constexpr int kTsBm = kTsAm + PT * PT * 4;
  static constexpr int kTsFlag = kTsBm + PT * PT * 4;
  static constexpr int kTsN = kTsFlag + 16;
  static constexpr int kTsMeta = kTsN + PT * PT * 4;
  static constexpr int kTStage = (kTsMeta + (int)sizeof(UnitMeta) + 127) & ~127;
  // regions
  static constexpr int kSStages0 = 0;
  static constexpr int kTStages0 = kSStages0 + kSStages * kSStage;
  // the producer's ring of unit words, kMetaRing entries of MetaEnt
  static constexpr int kMetas = kTStages0 + kTStages * kTStage;
  // barriers: sfull[2] sempty[2] tfull[3] pfull[3] tempty[3]
  static constexpr int kBars = kMetas + kMetaRing * 64;
  static constexpr int kNumBars = 2 * kSStages + 3 * kTStages;
  static constexpr int kAbort = kBars + kNumBars * 8;
  static constexpr int kTotal = kAbort + 16 + 1024;  // + alignment slack
};
static_assert(PipeLayout::kTotal <= 227 * 1024, "verify pipeline shared memory");
static_assert(kPrepChanBar + 2 * (PipeRoles<true>::kGroups - 1) <= 15,
              "the prep groups' named barrier ids (0 is the CTA barrier)");
static_assert(R::kBytes % 16 == 0, "records must keep 16-byte alignment");
static_assert(PipeLayout::kTsRk % 16 == 0 && PipeLayout::kTsFrag % 16 == 0,
              "token stage parts must keep 16-byte alignment");
static_assert(PipeLayout::kTStages0 % 128 == 0 && PipeLayout::kTStage % 128 == 0 &&
                  (PipeLayout::kTsRec + R::kA * 2) % 128 == 0 &&
                  (PipeLayout::kTsRec + R::kQ * 2) % 128 == 0 &&
                  (PipeLayout::kTsRec + R::kV * 2) % 128 == 0 &&
                  PipeLayout::kTsRv % 128 == 0 && PipeLayout::kTsRk % 128 == 0 &&
                  (PipeLayout::kTsRk + kDepthMax * PD * 2) % 128 == 0 &&
                  PipeLayout::kSStage % 1024 == 0 && PipeLayout::kTStages0 % 1024 == 0,
              "TMA destinations: 128-byte boundaries (1024 for the swizzled state)");

struct Bars {
  uint64_t *sfull, *sempty, *tfull, *pfull, *tempty;
  __device__ explicit Bars(unsigned char *smb) {
    uint64_t *b = reinterpret_cast<uint64_t *>(smb + PipeLayout::kBars);
    sfull = b;
    sempty = b + kSStages;
    tfull = b + 2 * kSStages;
    pfull = tfull + kTStages;
    tempty = pfull + kTStages;
  }
};

// ------------------------------------------------------------ mbarriers
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}"
               :: "r"(umma::smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}"
      :: "r"(umma::smem_u32(bar)), "r"(bytes) : "memory");
}
// This thread's cp.async copies so far (none, in this kernel) arrive on an
// mbarrier (counted in its expected arrivals) once they land.
__device__ __forceinline__ void cp_async_arrive(uint64_t *bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];"
               :: "r"(umma::smem_u32(bar)) : "memory");
}
// Use k of a barrier that completes once per use: every lane of the warp
// waits for use k (parity k & 1), and the warp agrees on the outcome, so a
// warp never splits over a shuffle or an MMA.  Bounded; on running out the
// warp sets the CTA's abort flag and the error bit and returns false.
__device__ __forceinline__ bool pipe_wait(uint64_t *bar, int use, int limit,
                                          volatile int *abort_flag, unsigned *err) {
  const bool ok = __all_sync(kFull, umma::mbar_wait(bar, (uint32_t)(use & 1), limit));
  if (!ok && (threadIdx.x & 31) == 0) {
    *abort_flag = 1;
    set_error(err, KDA_DERR_TIMEOUT);
  }
  return ok;
}
// Whether the CTA is stopping, agreed by the warp.
__device__ __forceinline__ bool stopping(volatile int *abort_flag) {
  return __any_sync(kFull, *abort_flag != 0);
}
__device__ __forceinline__ void named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ int named_and(int id, int n, int v) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.s32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\tselp.s32 %0, 1, 0, q;\n\t}"
      : "=r"(r) : "r"(v), "r"(id), "r"(n) : "memory");
  return r;
}
__device__ __forceinline__ int named_or(int id, int n, int v) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.s32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\tselp.s32 %0, 1, 0, q;\n\t}"
      : "=r"(r) : "r"(v), "r"(id), "r"(n) : "memory");
  return r;
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                         uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// a state pair (c, c+1) -> bf16x2 hi = rn(x), lo = rn(x - hi), c in the low half
__device__ __forceinline__ void split_pair(f2 x, uint32_t &hi, uint32_t &lo) {
  float a, b;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(x));
  umma::split_bf16x2(a, b, hi, lo);
}

// --------------------------------------------------------------- producer
// The words of units b0 .. b0 + 31 of this CTA (n = b0 + lane), one unit per
// lane, into the meta ring (entry n % kMetaRing), which only the producer
// reads.  Round one: slot, segment and row kind -- all a state copy needs.
__device__ void fetch_batch_a(const VerifyParams &p, unsigned char *smb, int b0, int cnt,
                              int lane) {
  typedef PipeLayout L;
  const int n = b0 + lane;
  if (n < cnt) {
    MetaEnt e = {};
    UnitMeta &m = e.m;
    const int H = p.H, u = blockIdx.x + n * gridDim.x, i = u / H;
    int c0 = 0, c1 = 0;
    m.slot = p.state_slots[i];
    if (p.mode == 0) {
      c0 = p.cu_seqlens[i];
      c1 = p.cu_seqlens[i + 1];
      m.spec = p.is_spec ? (p.is_spec[i] != 0) : 1;
    }
    int bad = 0;
    if (m.slot < 0 || m.slot >= p.P) bad = KDA_DERR_SLOT;
    if (p.mode == 0 && !bad) {
      if (c0 < 0 || c1 < c0 || c1 > p.N) {
        bad = KDA_DERR_SEGMENT;
      } else {
        m.tok0 = c0;
        m.T = c1 - c0;
        if (m.T > p.max_T || (m.spec && m.T > p.depth)) bad = KDA_DERR_DEPTH;
      }
    }
    if (bad) {
      set_error(p.err, (unsigned)bad);
      m.skip = 1;
      m.T = 0;
    }
    reinterpret_cast<MetaEnt *>(smb + L::kMetas)[n % kMetaRing] = e;
  }
  __syncwarp();
}

// Round two: the ring word and the beta values the unit's stages need, in
// two halves, so that the loads can be in flight while the first copies are
// issued (they would otherwise queue behind those copies' bytes).  The
// loads, into the lane's registers:
struct WordsB {
  int2 c;
  unsigned short bv[16];
};
__device__ __forceinline__ WordsB load_words_b(const VerifyParams &p, unsigned char *smb,
                                               int b0, int cnt, int lane) {
  typedef PipeLayout L;
  WordsB w;
  w.c = make_int2(0, 0);
#pragma unroll
  for (int q = 0; q < 16; ++q) w.bv[q] = 0;
  const int n = b0 + lane;
  if (n < cnt) {
    const UnitMeta m = reinterpret_cast<const MetaEnt *>(smb + L::kMetas)[n % kMetaRing].m;
    if (!m.skip) {
      const int H = p.H, u = blockIdx.x + n * gridDim.x, h = u - (u / H) * H;
      const size_t unit = (size_t)m.slot * H + h;
      w.c = *reinterpret_cast<const int2 *>(p.ctrl + unit * 2);
      const unsigned short *rb = reinterpret_cast<const unsigned short *>(p.rb) + unit * p.depth;
      const unsigned short *tb = reinterpret_cast<const unsigned short *>(p.beta);
#pragma unroll
      for (int q = 0; q < kDepthMax; ++q) w.bv[q] = q < p.depth ? rb[q] : 0;
#pragma unroll
      for (int q = 0; q < PT; ++q)
        w.bv[kDepthMax + q] = q < m.T ? tb[(size_t)(m.tok0 + q) * H + h] : 0;
    }
  }
  return w;
}
// ... and their checks and placement in the unit's meta ring entry.
__device__ __forceinline__ void place_words_b(const VerifyParams &p, unsigned char *smb, int b0,
                                              int cnt, int lane, const WordsB &w) {
  typedef PipeLayout L;
  const int n = b0 + lane;
  if (n < cnt) {
    MetaEnt &e = reinterpret_cast<MetaEnt *>(smb + L::kMetas)[n % kMetaRing];
    UnitMeta &m = e.m;
    if (!m.skip) {
      const bool ok = w.c.x >= 0 && w.c.x <= p.depth && w.c.y >= 0 && w.c.y <= w.c.x;
#pragma unroll
      for (int q = 0; q < 16; ++q) e.b[q] = w.bv[q];
      if (!ok) {
        set_error(p.err, KDA_DERR_RING);
        m.skip = 1;
        m.T = 0;
      } else {
        m.acc = w.c.y;
      }
    }
  }
  __syncwarp();
}
__device__ __forceinline__ void fetch_batch_b(const VerifyParams &p, unsigned char *smb, int b0,
                                              int cnt, int lane) {
  const WordsB w = load_words_b(p, smb, b0, cnt, lane);
  place_words_b(p, smb, b0, cnt, lane, w);
}

__device__ __forceinline__ void fetch_batch(const VerifyParams &p, unsigned char *smb, int b0,
                                            int cnt, int lane) {
  fetch_batch_a(p, smb, b0, cnt, lane);
  fetch_batch_b(p, smb, b0, cnt, lane);
}

__device__ __forceinline__ const MetaEnt &meta_of(unsigned char *smb, int n) {
  return reinterpret_cast<const MetaEnt *>(smb + PipeLayout::kMetas)[n % kMetaRing];
}

// L2 hint for unit n's state (lane 0).
__device__ __forceinline__ void prefetch_state(const VerifyParams &p, unsigned char *smb,
                                               int n, int lane) {
  const MetaEnt &e = meta_of(smb, n);
  if (lane == 0 && !e.m.skip) {
    const int u = blockIdx.x + n * gridDim.x, h = u - (u / p.H) * p.H;
    umma::prefetch_l2(p.pool + ((size_t)e.m.slot * p.H + h) * PD * PD, PD * PD * 4);
  }
}

// Unit n's state into state stage n % 2: one 64 KiB tensor copy (lane 0)
// completing on the stage's barrier, after the meta.
__device__ void issue_state(const VerifyParams &p, const CUtensorMap *smap, unsigned char *smb,
                            const Bars &bars, int n, int lane) {
  typedef PipeLayout L;
  const int s = n % kSStages;
  unsigned char *ss = smb + L::kSStages0 + s * L::kSStage;
  const UnitMeta m = meta_of(smb, n).m;
  if (lane == 0) {
    *reinterpret_cast<UnitMeta *>(ss + L::kSsMeta) = m;
    if (m.skip) {
      mbar_arrive(&bars.sfull[s]);
    } else {
      mbar_arrive_tx(&bars.sfull[s], PD * PD * 4);
      const int u = blockIdx.x + n * gridDim.x, h = u - (u / p.H) * p.H;
      const int row0 = (m.slot * p.H + h) * PD;  // the unit's first value row
      asm volatile(
          "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
          " [%0], [%1, {%2, %3, %4}], [%5];"
          :: "r"(umma::smem_u32(ss + L::kSsState)), "l"(reinterpret_cast<uint64_t>(smap)),
             "r"(0), "r"(row0), "r"(0), "r"(umma::smem_u32(&bars.sfull[s]))
          : "memory");
    }
  }
  __syncwarp();
}

// Unit n's tokens and pending ring entries into token stage n % 3: 16-byte
// async copies spread over the lanes (each lane's copies arrive on the
// stage's barrier when they land); the beta values and the meta by plain
// stores, lane 0 arriving after them.
// One TMA box of the map at (0, y, z) into shared memory, on `bar`.
__device__ __forceinline__ void tma_box3(uint32_t dst, const CUtensorMap *map, int y, int z,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];"
      :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// Unit n's token rows into token stage n % 3 (lane 0): one TMA box of PT
// tokens per field, their bytes on the stage's barrier.  Rows past the
// segment are other tokens or zeros and are never read.  Needs only the
// unit's segment, so the first unit's rows go out before the ring words are
// placed.
__device__ void issue_rows(const TokMaps *tmaps, unsigned char *smb, const Bars &bars, int n,
                           int H, int lane) {
  typedef PipeLayout L;
  const int k = n % kTStages;
  const UnitMeta m = meta_of(smb, n).m;
  if (m.skip || m.T == 0 || lane != 0) return;
  const int u = blockIdx.x + n * gridDim.x, h = u - (u / H) * H;
  const uint32_t base = umma::smem_u32(smb + L::kTStages0 + k * L::kTStage);
  const uint32_t bar = umma::smem_u32(&bars.tfull[k]);
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;"
               :: "r"(bar), "r"(4 * tmaps->tok_rows * PD * 2) : "memory");
  tma_box3(base + L::kTsRec + R::kK * 2, &tmaps->k, h, m.tok0, bar);
  tma_box3(base + L::kTsRec + R::kA * 2, &tmaps->a, h, m.tok0, bar);
  tma_box3(base + L::kTsRec + R::kQ * 2, &tmaps->q, h, m.tok0, bar);
  tma_box3(base + L::kTsRec + R::kV * 2, &tmaps->v, h, m.tok0, bar);
}

// The rest of unit n's stage: (unless `rows_done`) its token rows, its
// pending ring entries (k, alpha, v: one TMA box of the ring's depth entries
// each), the beta values and the meta by plain
// stores, lane 0 arriving after them.
__device__ void issue_tokens(const VerifyParams &p, const TokMaps *tmaps, unsigned char *smb,
                             const Bars &bars, int n, int lane, bool rows_done) {
  typedef PipeLayout L;
  const int k = n % kTStages;
  unsigned char *ts = smb + L::kTStages0 + k * L::kTStage;
  const MetaEnt &e = meta_of(smb, n);
  const UnitMeta m = e.m;
  if (!rows_done) issue_rows(tmaps, smb, bars, n, p.H, lane);
  if (!m.skip) {
    const int u = blockIdx.x + n * gridDim.x, h = u - (u / p.H) * p.H;
    const int unit = m.slot * p.H + h;
    if (m.acc > 0 && lane == 0) {
      const uint32_t base = umma::smem_u32(ts);
      const uint32_t bar = umma::smem_u32(&bars.tfull[k]);
      asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;"
                   :: "r"(bar), "r"(3 * tmaps->ring_rows * PD * 2) : "memory");
      tma_box3(base + L::kTsRk, &tmaps->rk, 0, unit, bar);
      tma_box3(base + L::kTsRk + kDepthMax * PD * 2, &tmaps->ra, 0, unit, bar);
      tma_box3(base + L::kTsRv, &tmaps->rv, 0, unit, bar);
    }
    if (lane < m.acc) reinterpret_cast<unsigned short *>(ts + L::kTsRb)[lane] = e.b[lane];
    if (lane >= 8 && lane < 8 + m.T)
      reinterpret_cast<unsigned short *>(ts + L::kTsRec)[R::kB + (lane - 8)] = e.b[lane];
  }
  if (lane == 0) *reinterpret_cast<UnitMeta *>(ts + L::kTsMeta) = m;
  cp_async_arrive(&bars.tfull[k]);  // this lane has no copies of its own in flight
  __syncwarp();
  if (lane == 0) mbar_arrive(&bars.tfull[k]);
}

// Whether use k of a barrier has completed, without waiting; agreed by the
// warp (every lane tests, so every lane that goes on has acquired it).
__device__ __forceinline__ bool use_done(uint64_t *bar, int use) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done) : "r"(umma::smem_u32(bar)), "r"((uint32_t)(use & 1)) : "memory");
  return __all_sync(kFull, done != 0);
}

// The producer issues each copy as soon as its stage is free, the state
// copies and the token copies independently of each other: unit n's state
// once the consumers have taken unit n - 2's state into registers, unit n's
// tokens once they have finished unit n - 3.  Polling is bounded: `limit`
// rounds with nothing to issue end the CTA's work with KDA_DERR_TIMEOUT.
__device__ void producer(const VerifyParams &p, const CUtensorMap *smap, const TokMaps *tmaps,
                         unsigned char *smb, int lane, int limit) {
  typedef PipeLayout L;
  const Bars bars(smb);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smb + L::kAbort);
  const int units = p.B * p.H, G = gridDim.x, u0 = blockIdx.x;
  const int cnt = u0 < units ? (units - u0 + G - 1) / G : 0;
  int s_last[kSStages], t_last[kTStages];  // last use issued of each stage
  for (int i = 0; i < kSStages; ++i) s_last[i] = -1;
  for (int i = 0; i < kTStages; ++i) t_last[i] = -1;
  // the first batch's slots; their ring words and beta values requested
  // before the first unit's state and rows go out, and placed after (units
  // 0 and 1 were hinted into L2 before the wait)
  int ns = 0, nt = 0, fetched = 0;
  fetch_batch_a(p, smb, 0, cnt, lane);
  const WordsB w0 = load_words_b(p, smb, 0, cnt, lane);  // in flight meanwhile
  // every copy takes the producer a while to issue: the first unit's state
  // and rows now, its ring entries as soon as its words are placed, and only
  // then the later units' copies
  const int early = cnt > 0 ? 1 : 0;  // stages whose rows went out here
  if (cnt > 0) {
    issue_state(p, smap, smb, bars, 0, lane);
    s_last[0] = 0;
    ns = 1;
    issue_rows(tmaps, smb, bars, 0, p.H, lane);
  }
  place_words_b(p, smb, 0, cnt, lane, w0);
  fetched = cnt < kMetaBatch ? cnt : kMetaBatch;
  int idle = 0;
  while (ns < cnt || nt < cnt) {
    if (stopping(abort_flag)) break;
    bool did = false;
    if (nt < cnt && nt < fetched && (nt < kTStages ||
                                     use_done(&bars.tempty[nt % kTStages], nt / kTStages - 1))) {
      issue_tokens(p, tmaps, smb, bars, nt, lane, nt < early);
      t_last[nt % kTStages] = nt / kTStages;
      ++nt;
      did = true;
    }
    if (ns < cnt && ns < fetched && (ns < kSStages ||
                                     use_done(&bars.sempty[ns % kSStages], ns / kSStages - 1))) {
      issue_state(p, smap, smb, bars, ns, lane);
      s_last[ns % kSStages] = ns / kSStages;
      if (ns + 1 < fetched) prefetch_state(p, smb, ns + 1, lane);
      ++ns;
      did = true;
    }
    // the next batch of words, once both streams are past the older half of
    // the meta ring
    if (fetched < cnt && (ns < nt ? ns : nt) >= fetched - kMetaBatch) {
      fetch_batch(p, smb, fetched, cnt, lane);
      fetched = fetched + kMetaBatch < cnt ? fetched + kMetaBatch : cnt;
      did = true;
    }
    if (did) {
      idle = 0;
    } else if (++idle > limit) {
      if (lane == 0) {
        *abort_flag = 1;
        set_error(p.err, KDA_DERR_TIMEOUT);
      }
      break;
    } else {
      __nanosleep(64);
    }
  }
  // stages whose rows went out early but whose tokens were not issued (the
  // CTA stopped first) get the rest of their copies and arrivals, so that
  // their barriers complete and can be drained
  for (; nt < early; ++nt) {
    issue_tokens(p, tmaps, smb, bars, nt, lane, true);
    t_last[nt % kTStages] = nt / kTStages;
  }
  // copies still in flight land before the CTA may exit (normally the
  // consumers have already waited for them)
  if (lane == 0) {
    for (int i = 0; i < kSStages; ++i)
      if (s_last[i] >= 0 &&
          !umma::mbar_wait(&bars.sfull[i], (uint32_t)(s_last[i] & 1), kDrainWaitPolls))
        set_error(p.err, KDA_DERR_UNSAFE);
    for (int i = 0; i < kTStages; ++i)
      if (t_last[i] >= 0 &&
          !umma::mbar_wait(&bars.tfull[i], (uint32_t)(t_last[i] & 1), kDrainWaitPolls))
        set_error(p.err, KDA_DERR_UNSAFE);
  }
  __syncwarp();
}

// ------------------------------------------------------------------- prep
// Projection-space tokens (RAW): a unit's rows are prepared in place before
// anything reads them -- the key L2-normalised over its 128 channels,
// alpha = 1 / (1 + e^z), beta = sigmoid(b) -- in IEEE fp32 and rounded to
// bf16 once, so decode, the drafts and the ring entries share those bits.
// The squared norm is always summed in one order: channel-pair sums
// fma(k_2p, k_2p, k_2p+1^2), a 32-lane xor tree over pairs 0..31 and one over
// pairs 32..63, then the two halves added; both routines below keep it, so a
// token prepared as an ordinary row or as a draft gets the same bits.
__device__ __forceinline__ float pair_sq(float2 k) { return fmaf(k.x, k.x, k.y * k.y); }
__device__ __forceinline__ float lane_tree(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(kFull, x, o);
  return x;
}
__device__ __forceinline__ float inv_norm(float half0, float half1) {
  return 1.f / fmaxf(sqrtf(half0 + half1), 1e-12f);
}
__device__ __forceinline__ float alpha_of_logit(float z) {
  return __frcp_rn(1.f + expf(z));
}
__device__ __forceinline__ float beta_of_logit(float b) {
  return __frcp_rn(1.f + expf(-b));
}
__device__ __forceinline__ float2 round_pair(float2 x, bf16 *dst) {
  const __nv_bfloat162 r = __floats2bfloat162_rn(x.x, x.y);
  *reinterpret_cast<__nv_bfloat162 *>(dst) = r;
  return __bfloat1622float2(r);
}

// Rows of a unit with no drafts (ordinary decode): prep math warp w
// prepares rows w, w + 2, ...; lane l holds channel pairs l and l + 32.
__device__ __forceinline__ void prep_raw_rows(bf16 *rec, int T, int w, int lane) {
  for (int t = w; t < T; t += kPrepMath / 32) {
    bf16 *r = rec + t * R::kStride;
    const int c0 = 2 * lane, c1 = 2 * lane + PD / 2;
    const float2 k0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(r + R::kK + c0));
    const float2 k1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(r + R::kK + c1));
    const float2 z0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(r + R::kA + c0));
    const float2 z1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(r + R::kA + c1));
    const float inv = inv_norm(lane_tree(pair_sq(k0)), lane_tree(pair_sq(k1)));
    round_pair(make_float2(k0.x * inv, k0.y * inv), r + R::kK + c0);
    round_pair(make_float2(k1.x * inv, k1.y * inv), r + R::kK + c1);
    round_pair(make_float2(alpha_of_logit(z0.x), alpha_of_logit(z0.y)), r + R::kA + c0);
    round_pair(make_float2(alpha_of_logit(z1.x), alpha_of_logit(z1.y)), r + R::kA + c1);
    if (lane == 0)
      rec[R::kB + t] = __float2bfloat16_rn(beta_of_logit(__bfloat162float(rec[R::kB + t])));
  }
}

// The third prep warp appends each unit's drafted inputs to the ring once
// the unit's products are handed over (pfull), outside the other two prep
// warps' barriers, so they start the next unit at once.
__device__ void ring_append(const VerifyParams &p, unsigned char *smb, int lane, int limit) {
  typedef PipeLayout L;
  const Bars bars(smb);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smb + L::kAbort);
  const int units = p.B * p.H, G = gridDim.x;
  const int cnt = (int)blockIdx.x < units ? (units - (int)blockIdx.x + G - 1) / G : 0;
  for (int n = 0; n < cnt; ++n) {
    const int k = n % kTStages;
    if (stopping(abort_flag)) break;
    if (!pipe_wait(&bars.pfull[k], n / kTStages, limit, abort_flag, p.err)) break;
    unsigned char *ts = smb + L::kTStages0 + k * L::kTStage;
    const UnitMeta m = *reinterpret_cast<const UnitMeta *>(ts + L::kTsMeta);
    if (!m.skip && m.spec && m.T > 0) {
      // entries 0..T-1 <- the drafted inputs (k, alpha, v, beta); this
      // unit's pending entries were copied out with the stage
      const int u = blockIdx.x + n * G, h = u - (u / p.H) * p.H;
      const size_t unit = (size_t)m.slot * p.H + h;
      const bf16 *rec = reinterpret_cast<const bf16 *>(ts + L::kTsRec);
      bf16 *wk = reinterpret_cast<bf16 *>(p.rk) + unit * p.depth * PD;
      bf16 *wa = reinterpret_cast<bf16 *>(p.ra) + unit * p.depth * PD;
      bf16 *wvr = reinterpret_cast<bf16 *>(p.rv) + unit * p.depth * PD;
      constexpr int CH = PD / 8;  // 16-byte chunks per vector
      for (int idx = lane; idx < m.T * 3 * CH; idx += 32) {
        const int t = idx / (3 * CH), r = idx - t * 3 * CH;
        const int which = r / CH, ch = r - which * CH;
        const int off = which == 0 ? R::kK : which == 1 ? R::kA : R::kV;
        bf16 *dst = (which == 0 ? wk : which == 1 ? wa : wvr) + (size_t)t * PD + ch * 8;
        *reinterpret_cast<uint4 *>(dst) =
            *reinterpret_cast<const uint4 *>(rec + t * R::kStride + off + ch * 8);
      }
      if (lane < m.T)
        reinterpret_cast<bf16 *>(p.rb)[unit * p.depth + lane] = rec[R::kB + lane];
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars.tempty[k]);
  }
}

// The drafts' operands of units grp, grp + PipeRoles<RAW>::kGroups, ..., by prep group
// grp's two channel-pair warps (pt < 64).  Every group walks every unit in
// order: it waits for each unit's token stage and arrives on its release
// (tempty), working only on its own units.  A parity wait cannot tell a
// stage barrier's phase from the one two after it; with every group among
// the releases, no stage is refilled before each group has seen its
// previous use, so no group's wait is ever two phases behind.
template <bool RAW>
__device__ void prep(const VerifyParams &p, unsigned char *smb, int pt, int grp, int limit) {
  const int bar = kPrepBar + 2 * grp, chan_bar = kPrepChanBar + 2 * grp;
  typedef PipeLayout L;
  const Bars bars(smb);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smb + L::kAbort);
  const int units = p.B * p.H, G = gridDim.x, lane = pt & 31;
  const int cnt = (int)blockIdx.x < units ? (units - (int)blockIdx.x + G - 1) / G : 0;
  for (int n = 0; n < cnt; ++n) {
    const int k = n % kTStages;
    const int u = blockIdx.x + n * G, h = u - (u / p.H) * p.H;
    // both prep warps take the same decision before any named barrier
    bool go = !stopping(abort_flag);
    if (go) go = pipe_wait(&bars.tfull[k], n / kTStages, limit, abort_flag, p.err);
    if (!named_and(bar, kPrepMath, go)) break;
    if (n % PipeRoles<RAW>::kGroups != grp) {  // another group's unit: only its release
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.tempty[k]);
      continue;
    }
    unsigned char *ts = smb + L::kTStages0 + k * L::kTStage;
    const UnitMeta m = *reinterpret_cast<const UnitMeta *>(ts + L::kTsMeta);
    const bool drafts = !m.skip && m.spec && m.T > 0;
    if (RAW && !m.skip && !drafts && m.T > 0) {  // drafts: prepared in the first phase
      prep_raw_rows(reinterpret_cast<bf16 *>(ts + L::kTsRec), m.T, pt >> 5, lane);
      named_sync(bar, kPrepMath);
    }
    if (drafts) {
      const bf16 *rec = reinterpret_cast<const bf16 *>(ts + L::kTsRec);
      unsigned char *fragb = ts + L::kTsFrag;
      float *am = reinterpret_cast<float *>(ts + L::kTsAm);
      float *bmat = reinterpret_cast<float *>(ts + L::kTsBm);
      float *nm = reinterpret_cast<float *>(ts + L::kTsN);
      const int T = m.T;
      // thread: value / key channels c, c + 1 (c = 2 pt), every drafted row:
      // gamma_t = prod_{r<=t} alpha_r, K~ = gamma k, Q~ = gamma q (zero past
      // T), K^ = k / gamma; fragments of the three (the thread fills half of
      // each 16-byte fragment entry)
      const int c = 2 * pt, f = c >> 4, fq = (c >> 2) & 3, half = (c >> 1) & 1;
      auto put = [&](int region, int t, float x, float y) {
        uint32_t hi, lo;
        umma::split_bf16x2(x, y, hi, lo);
        uint32_t *e = reinterpret_cast<uint32_t *>(fragb + region * 4096 +
                                                   ((f * 32) + 4 * t + fq) * 16);
        e[half] = hi;
        e[2 + half] = lo;
      };
      auto ld2 = [&](const bf16 *q) {
        return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(q));
      };
      int unsafe = 0;
      float2 kt[PT], qt[PT];
      const bool chan = pt < PD / 2;  // every math thread holds a channel pair
      if (chan) {
        // every load first (the stores below could alias them for the
        // compiler), then gamma, K~, Q~, K^ and their fragments
        // (all PT rows are loaded -- the stage holds them, past T other
        // tokens or stale bytes -- and the rows past T replaced after, so
        // no load waits on a branch)
        float2 av[PT], kv[PT], qv[PT];
#pragma unroll
        for (int t = 0; t < PT; ++t) {
          const bf16 *rr = rec + t * R::kStride;
          av[t] = ld2(rr + R::kA + c);
          kv[t] = ld2(rr + R::kK + c);
          qv[t] = ld2(rr + R::kQ + c);
        }
#pragma unroll
        for (int t = 0; t < PT; ++t) {
          if (t >= T) {
            av[t] = make_float2(1.f, 1.f);
            kv[t] = qv[t] = make_float2(0.f, 0.f);
          }
        }
        if (RAW) {
          // projection-space rows: the squared key norms (this warp's half of
          // the channel pairs) to the scratch, then the prepared, rounded k
          // and alpha of this pair in place and in registers
          float *nh = am;  // the pair products are written later
#pragma unroll
          for (int t = 0; t < PT; ++t) {
            const float x = lane_tree(pair_sq(kv[t]));
            if (lane == 0) nh[(pt >> 5) * PT + t] = x;
          }
          named_sync(chan_bar, 2 * 32);
          bf16 *rw = const_cast<bf16 *>(rec);
#pragma unroll
          for (int t = 0; t < PT; ++t) {
            if (t < T) {
              const float inv = inv_norm(nh[t], nh[PT + t]);
              kv[t] = round_pair(make_float2(kv[t].x * inv, kv[t].y * inv),
                                 rw + t * R::kStride + R::kK + c);
              av[t] = round_pair(make_float2(alpha_of_logit(av[t].x), alpha_of_logit(av[t].y)),
                                 rw + t * R::kStride + R::kA + c);
            }
          }
        }
        float2 g = make_float2(1.f, 1.f);
#pragma unroll
        for (int t = 0; t < PT; ++t) {
          g.x *= av[t].x;
          g.y *= av[t].y;
          kt[t] = make_float2(g.x * kv[t].x, g.y * kv[t].y);
          qt[t] = make_float2(g.x * qv[t].x, g.y * qv[t].y);
          float2 kh = make_float2(0.f, 0.f);
          if (t < T) {
            kh = make_float2(__fdividef(kv[t].x, g.x), __fdividef(kv[t].y, g.y));
            unsafe |= !(fminf(g.x, g.y) >= 0x1p-60f && fmaxf(g.x, g.y) <= 0x1p60f);
          }
          put(0, t, kt[t].x, kt[t].y);
          put(1, t, qt[t].x, qt[t].y);
          put(2, t, kh.x, kh.y);
        }
      }
      if (RAW && pt < T) {  // the rows' beta
        bf16 *rb = const_cast<bf16 *>(rec) + R::kB + pt;
        *rb = __float2bfloat16_rn(beta_of_logit(__bfloat162float(*rb)));
      }
      unsafe = named_or(bar, kPrepMath, unsafe);
      if (!unsafe) {
        // the pair products on the tensor cores, one prep warp each:
        // D row s, column t = K^_s . K~_t (warp 0: A) or K^_s . Q~_t (B)
        const uint4 *frag = reinterpret_cast<const uint4 *>(fragb);
        const int w = pt >> 5;
        if (w < 2) {
        float dp[4] = {0.f, 0.f, 0.f, 0.f}, dq[4] = {0.f, 0.f, 0.f, 0.f};
        float dr[4] = {0.f, 0.f, 0.f, 0.f};
        uint4 fa[PD / 16], fb[PD / 16];
#pragma unroll
        for (int ff = 0; ff < PD / 16; ++ff) {
          fa[ff] = frag[(2 * 8 + ff) * 32 + lane];  // K^ rows s
          fb[ff] = frag[(w * 8 + ff) * 32 + lane];  // K~ or Q~
        }
#pragma unroll
        for (int ff = 0; ff < PD / 16; ++ff) {
          mma16816(dp, fa[ff].x, 0u, fa[ff].y, 0u, fb[ff].x, fb[ff].y);
          mma16816(dq, fa[ff].z, 0u, fa[ff].w, 0u, fb[ff].x, fb[ff].y);
          mma16816(dr, fa[ff].x, 0u, fa[ff].y, 0u, fb[ff].z, fb[ff].w);
        }
        float *dst = w == 0 ? am : bmat;
        const int sI = lane >> 2, t0p = 2 * (lane & 3);
        dst[t0p * PT + sI] = dp[0] + (dq[0] + dr[0]);
        dst[(t0p + 1) * PT + sI] = dp[1] + (dq[1] + dr[1]);
        }
      } else {
        // gamma left [2^-60, 2^60] somewhere (K^ may overflow): the pair
        // matrices with explicit decay products instead, A_ts = sum_c k_tc
        // k_sc prod_{s<w<=t} alpha_wc (s < t) and B_ts with q_t (s <= t);
        // 4 lanes per pair, a quarter of the channels each
        const int nb = T * (T + 1) / 2, npairs = T * T, rg = pt & 3;
        for (int base = 0; base < npairs * 4; base += kPrepMath) {
          const int pair = (base + pt) >> 2;
          float acc = 0.f;
          int t = 0, sI = 0;
          const bool valid = pair < npairs, isB = pair < nb;
          if (valid) {
            int r = isB ? pair : pair - nb;
            if (isB) {
              while (r >= t + 1) { r -= t + 1; ++t; }
            } else {
              t = 1;
              while (r >= t) { r -= t; ++t; }
            }
            sI = r;
            for (int cc = rg; cc < PD; cc += 4) {
              float pr = 1.f;
              for (int w = sI + 1; w <= t; ++w)
                pr *= __bfloat162float(rec[w * R::kStride + R::kA + cc]);
              const float x = __bfloat162float(rec[t * R::kStride + (isB ? R::kQ : R::kK) + cc]);
              acc = fmaf(x * __bfloat162float(rec[sI * R::kStride + R::kK + cc]), pr, acc);
            }
          }
          acc += __shfl_xor_sync(kFull, acc, 1);
          acc += __shfl_xor_sync(kFull, acc, 2);
          if (valid && rg == 0) {
            if (isB) bmat[t * PT + sI] = acc;
            else am[t * PT + sI] = acc;
          }
        }
      }
      named_sync(bar, kPrepMath);
      // N = B M with M = (I + L)^-1 diag(beta), L = diag(beta) A strictly
      // lower (the drafts' corrections are delta = M (v - S^T K~), so that
      // o = S^T Q~ + N (v - S^T K~)).  Row r of Y = B (I + L)^-1 solves
      // Y (I + L) = B: Y[r][s] = B[r][s] - sum_{t > s} Y[r][t] L[t][s], by
      // back substitution over the columns s = 7 .. 0, one thread per row and
      // no barrier inside; then N = Y diag(beta).
      if (pt < PT) {
        const int r = pt;
        // every load first: beta, L's strict lower triangle, B's row r
        float bt[PT], lv[PT * (PT - 1) / 2], br[PT], y[PT];
#pragma unroll
        for (int q = 0; q < PT; ++q) {
          bt[q] = q < T ? __bfloat162float(rec[R::kB + q]) : 0.f;
          br[q] = (q <= r && r < T) ? bmat[r * PT + q] : 0.f;
        }
#pragma unroll
        for (int t = 1, i = 0; t < PT; ++t)
#pragma unroll
          for (int q = 0; q < t; ++q, ++i) lv[i] = t < T ? bt[t] * am[t * PT + q] : 0.f;
        // column by column: once Y[r][t] is known it leaves every column
        // s < t at once, so the dependent chain is one FMA per column
#pragma unroll
        for (int t = PT - 1; t >= 0; --t) {
          y[t] = br[t];
#pragma unroll
          for (int q = 0; q < t; ++q) br[q] = fmaf(-y[t], lv[t * (t - 1) / 2 + q], br[q]);
        }
#pragma unroll
        for (int q = 0; q < PT; ++q) nm[r * PT + q] = y[q] * bt[q];
      }
      named_sync(bar, kPrepMath);
      // Q^ = Q~ - N K~ (fragments, over Q~'s) and W = N v (fp32, over K^'s):
      // o_t = (S^T Q^)_t + W_t
      float *wv = reinterpret_cast<float *>(fragb + 2 * 4096);
      if (chan) {
        // loads first: v of every drafted row, N's lower triangle
        float2 vv[PT];
        float nn[PT * (PT + 1) / 2];
#pragma unroll
        for (int u = 0; u < PT; ++u) vv[u] = ld2(rec + u * R::kStride + R::kV + c);
#pragma unroll
        for (int u = 0; u < PT; ++u)
          if (u >= T) vv[u] = make_float2(0.f, 0.f);  // rows past T: other tokens
#pragma unroll
        for (int t = 0, i = 0; t < PT; ++t)
#pragma unroll
          for (int u = 0; u <= t; ++u, ++i) nn[i] = nm[t * PT + u];
#pragma unroll
        for (int t = 0, i = 0; t < PT; ++t) {
          float2 qh = qt[t], wt = make_float2(0.f, 0.f);
#pragma unroll
          for (int u = 0; u <= t; ++u, ++i) {
            qh.x = fmaf(-nn[i], kt[u].x, qh.x);
            qh.y = fmaf(-nn[i], kt[u].y, qh.y);
            wt.x = fmaf(nn[i], vv[u].x, wt.x);
            wt.y = fmaf(nn[i], vv[u].y, wt.y);
          }
          if (t >= T) qh = wt = make_float2(0.f, 0.f);
          put(1, t, qh.x, qh.y);
          *reinterpret_cast<float2 *>(wv + t * PD + c) = wt;
        }
      }
    }
    mbar_arrive(&bars.pfull[k]);
    if (!m.skip && pt == 0) {
      const size_t unit = (size_t)m.slot * p.H + h;
      int32_t *c = p.ctrl + unit * 2;
      c[0] = drafts ? m.T : 0;
      c[1] = 0;
    }
    // this warp is done with the stage
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars.tempty[k]);
  }
}

// -------------------------------------------------------------- consumers
template <bool RAW>
__device__ void consumer(const VerifyParams &p, unsigned char *smb, int tid, int limit) {
  typedef PipeLayout L;
  constexpr int F = PD / 16;
  const Bars bars(smb);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smb + L::kAbort);
  const int units = p.B * p.H, G = gridDim.x, H = p.H;
  const int lane = tid & 31, rg = tid & 3, j0 = 2 * (tid >> 2);
  const int cnt = (int)blockIdx.x < units ? (units - (int)blockIdx.x + G - 1) / G : 0;
  for (int n = 0; n < cnt; ++n) {
    const int s = n % kSStages, k = n % kTStages;
    const int u = blockIdx.x + n * G, h = u - (u / H) * H;
    if (stopping(abort_flag)) break;
    if (!pipe_wait(&bars.sfull[s], n / kSStages, limit, abort_flag, p.err)) break;
    f2 S[2][2 * F];
    {
      const unsigned char *ss = smb + L::kSStages0 + s * L::kSStage;
      if (!reinterpret_cast<const UnitMeta *>(ss + L::kSsMeta)->skip) {
        // chunk q = rg + 4f (key channels 4q .. 4q + 3) of rows j0, j0 + 1:
        // box q / 8, position (q % 8) ^ (row % 8) -- the eight rows of a
        // warp's lanes land in distinct bank groups
        const unsigned char *st = ss + L::kSsState;
#pragma unroll
        for (int f = 0; f < F; ++f) {
          const int q = rg + 4 * f, box = (q >> 3) * (PD * 32 * 4), cb = q & 7;
          const ulonglong2 x = *reinterpret_cast<const ulonglong2 *>(
              st + box + j0 * 128 + ((cb ^ (j0 & 7)) << 4));
          const ulonglong2 y = *reinterpret_cast<const ulonglong2 *>(
              st + box + (j0 + 1) * 128 + ((cb ^ ((j0 + 1) & 7)) << 4));
          S[0][2 * f] = x.x; S[0][2 * f + 1] = x.y;
          S[1][2 * f] = y.x; S[1][2 * f + 1] = y.y;
        }
      }
    }
    // the state stage is free again (its bytes are in registers)
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars.sempty[s]);
    // the unit's tokens and ring entries (the prep may still be working on
    // the drafts' fragments)
    if (!pipe_wait(&bars.tfull[k], n / kTStages, limit, abort_flag, p.err)) break;
    unsigned char *ts = smb + L::kTStages0 + k * L::kTStage;
    const UnitMeta m = *reinterpret_cast<const UnitMeta *>(ts + L::kTsMeta);
    const size_t unit = (size_t)m.slot * H + h;
    const bool drafts = !m.skip && m.spec && m.T > 0;
    const bf16 *rec = reinterpret_cast<const bf16 *>(ts + L::kTsRec);
    auto store_state = [&]() {
      ulonglong2 *c0 = reinterpret_cast<ulonglong2 *>(p.pool + unit * PD * PD + (size_t)j0 * PD);
      ulonglong2 *c1 = c0 + PD / 4;
#pragma unroll
      for (int f = 0; f < F; ++f) {
        c0[rg + 4 * f] = make_ulonglong2(S[0][2 * f], S[0][2 * f + 1]);
        c1[rg + 4 * f] = make_ulonglong2(S[1][2 * f], S[1][2 * f + 1]);
      }
    };
    if (!m.skip) {
      // lazy commit: replay the accepted ring entries
      const bf16 *rk = reinterpret_cast<const bf16 *>(ts + L::kTsRk);
      const bf16 *ra = rk + kDepthMax * PD;
      const bf16 *rv = reinterpret_cast<const bf16 *>(ts + L::kTsRv);
      const bf16 *rb = reinterpret_cast<const bf16 *>(ts + L::kTsRb);
      float o0 = 0.f, o1 = 0.f;
      for (int t = 0; t < m.acc; ++t)
        kda_step_ptrs<PD, false, bf16>(S, rk + t * PD, ra + t * PD, nullptr, rv + t * PD,
                                       rb + t, rg, j0, o0, o1);
    }
    if (!m.skip && m.spec && m.acc > 0) store_state();  // the committed state
    // projection-space rows are read only once the prep warps have prepared them
    if (RAW && !pipe_wait(&bars.pfull[k], n / kTStages, limit, abort_flag, p.err)) break;
    if (!m.skip && !m.spec) {
      // ordinary decode (or materialize): apply and commit
      float o0 = 0.f, o1 = 0.f;
      for (int t = 0; t < m.T; ++t) {
        kda_step_ptrs<PD, true, bf16>(S, rec + R::kK + t * PD, rec + R::kA + t * PD,
                                      rec + R::kQ + t * PD, rec + R::kV + t * PD,
                                      rec + R::kB + t, rg, j0, o0, o1);
        if (rg == 0)
          *reinterpret_cast<float2 *>(p.o + ((size_t)(m.tok0 + t) * H + h) * PD + j0) =
              make_float2(o0, o1);
      }
      if (m.acc > 0 || m.T > 0) store_state();
    }
    if (!RAW && !pipe_wait(&bars.pfull[k], n / kTStages, limit, abort_flag, p.err)) break;
    if (drafts) {
      // drafts: o_t = (S^T Q^)_t + W_t, S^T Q^ from the registers on the
      // tensor cores, hi*hi + lo*hi + hi*lo
      const uint4 *frag = reinterpret_cast<const uint4 *>(ts + L::kTsFrag) + 8 * 32;
      uint4 b[F];
#pragma unroll
      for (int f = 0; f < F; ++f) b[f] = frag[f * 32 + lane];
      float dz[4] = {0.f, 0.f, 0.f, 0.f}, ez[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int f = 0; f < F; ++f) {
        uint32_t ah[4], al[4];
        split_pair(S[0][2 * f], ah[0], al[0]);      // row g,   k 2r..2r+1
        split_pair(S[1][2 * f], ah[1], al[1]);      // row g+8, k 2r..2r+1
        split_pair(S[0][2 * f + 1], ah[2], al[2]);  // row g,   k 2r+8..
        split_pair(S[1][2 * f + 1], ah[3], al[3]);  // row g+8, k 2r+8..
        mma16816(dz, ah[0], ah[1], ah[2], ah[3], b[f].x, b[f].y);
        mma16816(ez, al[0], al[1], al[2], al[3], b[f].x, b[f].y);
        mma16816(ez, ah[0], ah[1], ah[2], ah[3], b[f].z, b[f].w);
      }
      // D row g / g + 8 = column j0 / j0 + 1, columns 2r, 2r + 1 = rows t
      const float *wv = reinterpret_cast<const float *>(ts + L::kTsFrag + 2 * 4096);
      const int t0 = 2 * rg;
      const float2 w0 = *reinterpret_cast<const float2 *>(wv + t0 * PD + j0);
      const float2 w1 = *reinterpret_cast<const float2 *>(wv + (t0 + 1) * PD + j0);
      if (t0 < m.T)
        *reinterpret_cast<float2 *>(p.o + ((size_t)(m.tok0 + t0) * H + h) * PD + j0) =
            make_float2(dz[0] + ez[0] + w0.x, dz[2] + ez[2] + w0.y);
      if (t0 + 1 < m.T)
        *reinterpret_cast<float2 *>(p.o + ((size_t)(m.tok0 + t0 + 1) * H + h) * PD + j0) =
            make_float2(dz[1] + ez[1] + w1.x, dz[3] + ez[3] + w1.y);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars.tempty[k]);
  }
}

template <bool RAW>
__global__ void __launch_bounds__(PipeRoles<RAW>::kThreads, 1)
    verify_pipe_kernel(const VerifyParams p, const __grid_constant__ CUtensorMap smap,
                       const __grid_constant__ TokMaps tmaps) {
  typedef PipeLayout L;
  extern __shared__ float4 smem4[];
  unsigned char *smb = umma::align1024(smem4);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int units = p.B * p.H;
  if (tid == 0) {
    const Bars b(smb);
    for (int i = 0; i < kSStages; ++i) {
      umma::mbar_init(&b.sfull[i], 1);
      umma::mbar_init(&b.sempty[i], kConsumerWarps);
    }
    for (int i = 0; i < kTStages; ++i) {
      umma::mbar_init(&b.tfull[i], 32 + 1);  // async arrivals of the lanes + lane 0
      umma::mbar_init(&b.pfull[i], kPrepMath);
      // per use: the consumers, every prep warp and the ring warp
      umma::mbar_init(&b.tempty[i], kConsumerWarps + PipeRoles<RAW>::kPrepWarps);
    }
    *reinterpret_cast<volatile int *>(smb + L::kAbort) = 0;
  }
  // Launched as a programmatic dependent of the previous kernel: until
  // griddepcontrol.wait returns, only the tensor-map descriptor prefetches
  // and L2 prefetch hints for this CTA's first
  // two units (state, ring word, ring beta, token rows), at the addresses the
  // slot table and segment offsets give when read (relaxed reads that the
  // previous kernel may still be writing: a stale value wastes a hint, and
  // L2 is where that kernel's writes become visible, so nothing stale is
  // used).
  if (warp == kProducerWarp) {
    // lanes 8 .. 15: the tensor maps' descriptors, which a copy otherwise
    // fetches at its first use, holding up the producer's first copies
    if (lane >= 8 && lane < 16) {
      const CUtensorMap *tm = lane == 8 ? &smap : &tmaps.k + (lane - 9);
      asm volatile("prefetch.tensormap [%0];"
                   :: "l"(reinterpret_cast<uint64_t>(tm)) : "memory");
    }
    // lanes 0, 1: the first two units' words and states; lanes 2, 3: their
    // token rows (k, alpha, v, q of each drafted position)
    const int n = lane & 1, u = blockIdx.x + n * gridDim.x;
    if (lane < 4 && u < units) {
      const int i = u / p.H, h = u - (u / p.H) * p.H;
      if (lane < 2) {
        int s0;
        asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];"
                     : "=r"(s0) : "l"(p.state_slots + i) : "memory");
        if (s0 >= 0 && s0 < p.P) {
          const size_t un = (size_t)s0 * p.H + h;
          umma::prefetch_l2(p.pool + un * PD * PD, PD * PD * 4);
          asm volatile("prefetch.global.L2 [%0];" :: "l"(p.ctrl + un * 2));
          asm volatile("prefetch.global.L2 [%0];"
                       :: "l"(reinterpret_cast<const bf16 *>(p.rb) + un * p.depth));
        }
      } else if (p.mode == 0) {
        int c0, c1;
        asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];"
                     : "=r"(c0) : "l"(p.cu_seqlens + i) : "memory");
        asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];"
                     : "=r"(c1) : "l"(p.cu_seqlens + i + 1) : "memory");
        if (c0 >= 0 && c1 >= c0 && c1 - c0 <= PT && c1 <= p.N) {
          for (int t = c0; t < c1; ++t) {
            const size_t row = ((size_t)t * p.H + h) * PD;
            umma::prefetch_l2(reinterpret_cast<const bf16 *>(p.k) + row, PD * 2);
            umma::prefetch_l2(reinterpret_cast<const bf16 *>(p.alpha) + row, PD * 2);
            umma::prefetch_l2(reinterpret_cast<const bf16 *>(p.v) + row, PD * 2);
            umma::prefetch_l2(reinterpret_cast<const bf16 *>(p.q) + row, PD * 2);
            asm volatile("prefetch.global.L2 [%0];"
                         :: "l"(reinterpret_cast<const bf16 *>(p.beta) + (size_t)t * p.H + h));
          }
        }
      }
    }
  }
  __syncthreads();
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int limit = p.spin_limit;
  if (warp == kProducerWarp) producer(p, &smap, &tmaps, smb, lane, limit);
  else if (warp == PipeRoles<RAW>::kRingWarp) ring_append(p, smb, lane, limit);
  else if (warp >= kPrepWarp0) {
    const int grp = (warp - kPrepWarp0) >> 1;
    prep<RAW>(p, smb, tid - 32 * (kPrepWarp0 + 2 * grp), grp, limit);
  }
  else consumer<RAW>(p, smb, tid, limit);
  __syncthreads();
}

}  // namespace

namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t,
                                  void *, const cuuint64_t *, const cuuint64_t *,
                                  const cuuint32_t *, const cuuint32_t *,
                                  CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled from the driver, looked up once.
EncodeTiledFn encode_tiled_fn() {
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

// The pool [P * H * PD value rows][PD key channels] fp32 as a 3-D tensor:
// x = key channel within a group of 32 (128 bytes), y = value row (stride
// PD * 4 bytes), z = group of 32 key channels (stride 128 bytes).  One box of
// 32 x PD x 4 is a unit's whole state, landing as four 16 KB blocks (one per
// group, z outermost) of 128-byte rows with the 128-byte swizzle: the same
// bytes four 2-D boxes of 32 channels x PD rows would give, in one copy.
cudaError_t state_map(CUtensorMap *tm, float *pool, int P, int H) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t gdim[3] = {32, (cuuint64_t)P * H * PD, PD / 32};
  const cuuint64_t gstride[2] = {(cuuint64_t)PD * 4, 128};
  const cuuint32_t box[3] = {32, (cuuint32_t)PD, PD / 32};
  const cuuint32_t estride[3] = {1, 1, 1};
  const CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, pool, gdim, gstride, box,
                         estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Packed bf16 tokens [N][H][PD] as a 3-D tensor map, boxes of PD channels x 1
// head x min(PT, N) tokens, zero fill past N.
cudaError_t token_map(CUtensorMap *tm, const void *base, int N, int H) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t gdim[3] = {(cuuint64_t)PD, (cuuint64_t)H, (cuuint64_t)N};
  const cuuint64_t gstride[2] = {(cuuint64_t)PD * 2, (cuuint64_t)H * PD * 2};
  const cuuint32_t box[3] = {(cuuint32_t)PD, 1, (cuuint32_t)(N < PT ? N : PT)};
  const cuuint32_t estride[3] = {1, 1, 1};
  const CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base),
                         gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// A ring payload array [units][depth][PD] (bf16) as a 3-D tensor map, boxes
// of PD channels x depth entries x 1 unit.
cudaError_t ring_map(CUtensorMap *tm, const void *base, int depth, int units) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t gdim[3] = {(cuuint64_t)PD, (cuuint64_t)depth, (cuuint64_t)units};
  const cuuint64_t gstride[2] = {(cuuint64_t)PD * 2, (cuuint64_t)depth * PD * 2};
  const cuuint32_t box[3] = {(cuuint32_t)PD, (cuuint32_t)depth, 1};
  const cuuint32_t estride[3] = {1, 1, 1};
  const CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base),
                         gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}
}  // namespace

bool verify_pipe_applies(const VerifyParams &p, kda_dtype dt, int D) {
  return D == PD && dt == KDA_BF16 && p.depth <= kDepthMax && p.max_T <= PT;
}

cudaError_t launch_verify_pipe(const VerifyParams &p, cudaStream_t s) {
  static std::mutex mu;
  static int sms_of[64] = {};
  static bool ready[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const size_t smem = PipeLayout::kTotal;
  int sms = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!ready[dev]) {
      cudaError_t e = cudaFuncSetAttribute(verify_pipe_kernel<false>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(verify_pipe_kernel<true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&sms_of[dev], cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) return e;
      ready[dev] = true;
    }
    sms = sms_of[dev];
  }
  const int units = p.B * p.H;
  if (units == 0 || sms < 1) return units == 0 ? cudaSuccess : cudaErrorInvalidDevice;
  // the fewest CTAs that keep the most units per CTA at ceil(units / SMs):
  // every CTA then walks the same number of units (give or take one)
  const int per = (units + sms - 1) / sms;
  const int grid = (units + per - 1) / per;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(p.raw ? PipeRoles<true>::kThreads : PipeRoles<false>::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  CUtensorMap smap;
  cudaError_t e = state_map(&smap, p.pool, p.P, p.H);
  if (e != cudaSuccess) return e;
  TokMaps tmaps;
  memset(&tmaps, 0, sizeof(tmaps));  // materialize: no tokens, never read
  tmaps.ring_rows = p.depth;
  tmaps.tok_rows = p.N < PT ? p.N : PT;
  e = ring_map(&tmaps.rk, p.rk, p.depth, p.P * p.H);
  if (e == cudaSuccess) e = ring_map(&tmaps.ra, p.ra, p.depth, p.P * p.H);
  if (e == cudaSuccess) e = ring_map(&tmaps.rv, p.rv, p.depth, p.P * p.H);
  if (e != cudaSuccess) return e;
  if (p.mode == 0 && p.N > 0) {
    e = token_map(&tmaps.k, p.k, p.N, p.H);
    if (e == cudaSuccess) e = token_map(&tmaps.a, p.alpha, p.N, p.H);
    if (e == cudaSuccess) e = token_map(&tmaps.q, p.q, p.N, p.H);
    if (e == cudaSuccess) e = token_map(&tmaps.v, p.v, p.N, p.H);
    if (e != cudaSuccess) return e;
  }
  return cudaLaunchKernelEx(&cfg, p.raw ? verify_pipe_kernel<true> : verify_pipe_kernel<false>,
                            p, smap, tmaps);
}

}  // namespace kda
