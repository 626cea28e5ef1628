// Pipelined tensor-memory (tcgen05) consumer for query-row groups of 17..64
// rows per KV head (MTP verify rows x GQA), dense paged decode on sm_103a.
//
// Warp roles (one CTA per SM; NWG = 2 or 4 softmax warpgroups):
//  * warps 0 .. 4 NWG - 1: the softmax warpgroups. TMEM lane quarter
//    q = warp % 4 holds stage tokens 32q..32q+31, so thread (warp, lane) owns
//    token 32q + lane; warpgroup w = warp / 4 owns query rows [w*RH, (w+1)*RH);
//  * warp 4 NWG: the producer of the tile kernel (page ids, TMA ring, Q ring);
//  * warp 4 NWG + 1: one thread issues every tcgen05.mma and commit.
// Four warpgroups of 16 rows put four softmax warps on each SM sub-partition
// (better latency hiding than two warpgroups of 32 rows) at 96 registers a
// thread.
//
// Per stage k (128 tokens), accumulators in tensor memory:
//   S^T[128 tok x RN]  = K . Q^T          (double-buffered: S(k+1) runs while
//                                          the softmax of stage k runs)
//   O^T[128 dims x RN] += V^T . P^T       (dims on lanes; one block per 128 dims)
//   L^T[64 x RN]       += 1 . P^T         (row sums from the same rounded P)
// The MMA thread issues S(k+1) before PV(k), so the tensor pipe computes the
// next scores and the previous products while the softmax warps work.
//
// Operands (128-byte swizzle):
//  * FP8 caches: S is kind::f8f6f4 with K read in place and Q as a three-term
//    e4m3 sum q = hi + mid + lo (each term rounded to 4 significant bits, the
//    last to nearest e4m3), accumulated into one S: about 12 significant bits
//    per query element. PV is kind::f16: the softmax warps convert the
//    stage's V to FP16 in place over the stage's K and V bytes (the per-token
//    V scale folded in, times 2^-4 so any scale up to 2048 fits FP16), and
//    P is FP16.
//  * BF16 caches: kind::f16 BF16 throughout, K and V read in place, P as a
//    two-term BF16 sum hi + lo (PV and L accumulate both).
//
// Softmax: a lazy reference max per row (m_r). P = 2^(s c_r - m_r) is taken
// against it; when a score exceeds its reference by more than 2^8 (always on
// a segment's first stage, rarely later) all softmax warps take a slow path
// that reduces the stage's row maxima, raises m_r and rescales the row's O
// and L columns in tensor memory. The warpgroups own disjoint columns, so a
// rescale never touches the other warpgroup's rows.
//
// Sources of the method: PR "Add paged-attention Tile kernel" (split-KV
// partials, per-tensor/per-token scales), PR "Extend packed D256 PA decode
// pipe to page16, transposed V and sliding windows" (scale before mask, MTP
// rows, windows), PR "Merge gfx1250 PA decode partitions in the tile kernel
// and speed up dense decode" (Dense tile kernels: MTP4 at GQA16, P kept next
// to its MMA, interior pages without masks; Partition merges). The warp roles,
// the tensor-memory layout and the operand splits are this implementation's.
#pragma once

#include "pa_tc.cuh"

namespace pa {
namespace dev {

constexpr int kMtpTT = 128;            // tokens per stage (M of S^T)
constexpr int kBarStage = 2;           // named barrier of all softmax threads (1 = merges)
constexpr int kBarWg0 = 3;             // 3, 4, ...: named barriers of one softmax warpgroup (128 threads)
constexpr float kVtokUnit = 0.0625f;   // per-token V scales enter FP16 V as vs * 2^-4

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
// RH consecutive 32-bit columns of this thread's TMEM lane.
template <int RH>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&v)[RH]) {
  static_assert(RH == 16 || RH == 32, "columns per load");
  if constexpr (RH == 32)
    tmem_ld32(taddr, v);
  else
    tmem_ld16(taddr, v);
}
template <int RH>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t (&v)[RH]) {
  if constexpr (RH == 32)
    tmem_st32(taddr, v);
  else
    tmem_st16(taddr, v);
}
__device__ __forceinline__ float4 lds128f(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ void sts32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t hmul2_bits(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Maxima over the warp's 32 lanes of RH per-lane values (one per row), with
// 31 shuffles: each butterfly step halves the values a lane holds, the lanes
// with the step's bit set keeping the upper half. Lane l ends with the maximum
// of row l % RH (v is overwritten).
template <int RH>
__device__ __forceinline__ float rowmax_transpose(float (&v)[RH], int lane) {
  if constexpr (RH == 16) {
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = fmaxf(v[j], __shfl_xor_sync(0xffffffffu, v[j], 16));
  }
#pragma unroll
  for (int half = RH / 2, b = RH / 2; half >= 1; half >>= 1, b >>= 1) {
    const bool upper = (lane & b) != 0;
#pragma unroll
    for (int j = 0; j < half; ++j) {
      const float send = upper ? v[j] : v[j + half];
      const float keep = upper ? v[j + half] : v[j];
      v[j] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, b));
    }
  }
  return v[0];
}

// Maximum of N values as a tree of three-input maxima (fixed bounds, so the
// temporaries stay in registers).
template <int N>
struct Max3Tree {
  __device__ __forceinline__ static float run(const float (&a)[N]) {
    constexpr int M = (N + 2) / 3;
    float b[M];
#pragma unroll
    for (int i = 0; i < M; ++i) {
      if (3 * i + 2 < N)
        b[i] = fmax3(a[3 * i], a[3 * i + 1], a[3 * i + 2]);
      else if (3 * i + 1 < N)
        b[i] = fmaxf(a[3 * i], a[3 * i + 1]);
      else
        b[i] = a[3 * i];
    }
    return Max3Tree<M>::run(b);
  }
};
template <>
struct Max3Tree<1> {
  __device__ __forceinline__ static float run(const float (&a)[1]) { return a[0]; }
};

// Pipeline barriers of the consumer (eight bytes each, from p.off_ubar).
struct MtpBars {
  uint32_t base;
  // S(k) in TMEM / S(k) read / P(k) and V(k) ready: one barrier per S^T
  // buffer, indexed k % SB
  __device__ __forceinline__ uint32_t s_full(int i) const { return base + 8u * i; }
  __device__ __forceinline__ uint32_t s_free(int i) const { return base + 24u + 8u * i; }
  __device__ __forceinline__ uint32_t p_full(int i) const { return base + 48u + 8u * i; }
  // PV(k) complete, three barriers indexed k % 3: between two observations
  // the softmax warps leave up to three PVs unobserved (their P buffers), so
  // no barrier may complete twice in that window
  __device__ __forceinline__ uint32_t pv_done(int i) const { return base + 72u + 8u * i; }
  __device__ __forceinline__ uint32_t q_ready() const { return base + 96u; }  // segment's Q operand written
  __device__ __forceinline__ uint32_t drained() const { return base + 104u; }  // every MMA complete
};

// NWG softmax warpgroups (warps 0 .. 4 NWG - 1) of RH rows each, then the
// producer warp and the MMA warp.
template <bool FP8, int D, bool VTOK, int RH, int NWG>
struct MtpCfg {
  static constexpr int TT = kMtpTT;
  static constexpr int RN = NWG * RH;            // rows of the MMA block (N of S^T and O^T)
  static constexpr int kSoftWarps = 4 * NWG;
  static constexpr int kSoft = 32 * kSoftWarps;  // softmax threads
  static constexpr int kThreads = kSoft + 64;
  static constexpr int kProducerWarp = kSoftWarps;
  static constexpr int kMmaWarp = kSoftWarps + 1;
  static constexpr int ELT = FP8 ? 1 : 2;
  static constexpr int NCH = D * ELT / 128;      // 128-byte chunks per token row of a stage
  static constexpr int DCH = D / 128;            // O^T blocks of 128 dims
  static constexpr int QTERMS = FP8 ? 3 : 1;
  static constexpr int QCH = FP8 ? D / 128 : D / 64;  // 128-byte chunks per query row of the Q operand
  static constexpr uint32_t kQTermBytes = (uint32_t)QCH * RN * 128u;
  // P^T slots of [128 tokens][128 B]: FP8 caches keep one FP16 term in three
  // buffers (P(k) is written while PV(k-1) and PV(k-2) may still read the
  // others); BF16 caches keep P as two BF16 terms hi + lo (about 16
  // significant bits) in one buffer.
  static constexpr int PT = FP8 ? 1 : 2;  // terms
  static constexpr int PB = FP8 ? 3 : 1;  // buffers
  static constexpr int NP = PT * PB;      // slots
  // S^T buffers: S(k) goes to buffer k % SB, so the MMA thread runs S up to
  // SB stages ahead of the slowest softmax warpgroup
  static constexpr int SB = 3;
  // tensor-memory columns
  static constexpr uint32_t kColS = 0;                   // S^T buffers: SB blocks of RN columns
  static constexpr uint32_t kColO = SB * RN;             // O^T: DCH blocks of RN columns
  static constexpr uint32_t kColL = (SB + DCH) * RN;     // L^T (M = 64 layout: lanes 0-15 of each quarter)
  static constexpr uint32_t kCols = kColL + RN <= 256 ? 256 : 512;  // a power of two (one CTA per SM)
  static_assert(kColL + RN <= kCols, "tensor memory budget");
  static_assert(!(D == 256 && RN > 32), "head_dim 256 takes at most 32 rows");
  // instruction descriptors (FP8 caches: S e4m3 x e4m3, PV and L FP16; BF16 caches: BF16)
  static constexpr uint32_t kIdS = umma_idesc_ab(!FP8, 128, RN, false, false);
  static constexpr uint32_t kIdPV = umma_idesc_ab(!FP8, 128, RN, true, true);
  static constexpr uint32_t kIdL = umma_idesc_ab(!FP8, 64, RN, false, true);
};

// Shared-memory regions of the consumer (byte offsets from the aligned base):
//   p.off_q16  Q operand: QTERMS x [QCH chunks][RN rows][128 B]
//   p.off_p16  P^T: NP slots of [128 tokens][128 B] (rows of warpgroup w at
//              bytes [w*RH*2, (w+1)*RH*2)), then the ones operand (2 KiB)
//   p.off_rows row state: c[64], m[64], pos[64], alpha[64], red[4][64]
template <bool FP8, int D, bool VTOK, int RH, int NWG>
struct MtpSoftmax {
  using C = MtpCfg<FP8, D, VTOK, RH, NWG>;
  static constexpr int TT = C::TT;
  static constexpr int RN = C::RN;

  const PaParams& p;
  Smem sm;
  MtpBars bars;
  int warp, lane, quarter, wg, tok;
  uint32_t tmem = 0, lane_addr = 0;
  float kscale = 1.f, vscale = 1.f;
  // The per-row score scales c_r and reference maxima m_r live in shared
  // memory (row_c, row_m) and are read with broadcast 128-bit loads.
  int n = 0;       // ring stages consumed
  int k = 0;       // stages with tokens (MMA stage index)
  int kd = 0;      // PV completions observed
  int nq = 0;      // Q ring slots consumed
  int seg_k0 = 0;  // k of the current segment's first stage with tokens
  bool ok = true;
  int Lseg = 0;

  __device__ __forceinline__ MtpSoftmax(const PaParams& p_, Smem s, uint32_t tm) : p(p_), sm(s) {
    bars.base = sm.base_u32 + p.off_ubar;
    warp = threadIdx.x >> 5;
    lane = threadIdx.x & 31;
    quarter = warp & 3;
    wg = warp >> 2;
    tok = 32 * quarter + lane;
    tmem = tm;
    lane_addr = (uint32_t)(32 * quarter) << 16;
    if (FP8 && p.scale_mode == kScalePerTensor) kscale = __ldg(p.k_scale);
    vscale = per_tensor_vscale(p) * (VTOK ? 1.f / kVtokUnit : 1.f);
  }

  __device__ __forceinline__ float* row_c() const { return reinterpret_cast<float*>(sm.base + p.off_rows); }
  __device__ __forceinline__ float* row_m() const { return row_c() + 64; }
  __device__ __forceinline__ int* row_pos() const { return reinterpret_cast<int*>(row_c() + 128); }
  __device__ __forceinline__ float* row_alpha() const { return row_c() + 192; }
  __device__ __forceinline__ float* row_red() const { return row_c() + 256; }  // [4 quarters][64]
  // shared-space addresses of the score scales and positions (explicit ld.shared in the hot loop)
  __device__ __forceinline__ uint32_t row_c_u32(int r) const { return sm.base_u32 + p.off_rows + 4u * (uint32_t)r; }
  __device__ __forceinline__ uint32_t row_m_u32(int r) const { return sm.base_u32 + p.off_rows + 256u + 4u * (uint32_t)r; }
  __device__ __forceinline__ uint32_t row_pos_u32(int r) const { return sm.base_u32 + p.off_rows + 512u + 4u * (uint32_t)r; }
  __device__ __forceinline__ uint32_t row_alpha_u32(int r) const { return sm.base_u32 + p.off_rows + 768u + 4u * (uint32_t)r; }
  __device__ __forceinline__ uint32_t q16() const { return sm.base_u32 + p.off_q16; }
  __device__ __forceinline__ uint32_t pslot(int i) const { return sm.base_u32 + p.off_p16 + (uint32_t)i * (TT * 128u); }

  __device__ __forceinline__ void fail() {
    ok = false;
    if (lane == 0) {
      flag_status(p, kStatusTimeout);
      sm.misc(p)[0] |= 1;
    }
  }

  // Wait until PV(x) has completed (completions are observed in order).
  __device__ __forceinline__ bool wait_pv(int x) {
    while (kd <= x) {
      if (!mbar_wait(bars.pv_done(kd % 3), (kd / 3) & 1)) {
        fail();
        return false;
      }
      ++kd;
    }
    tc_fence_after();
    return true;
  }

  // Build the segment's Q operand from the Q ring (rows past R are zeros),
  // the per-row score scale c_r and position, reset the reference max.
  // has_tokens: the segment's first stage holds tokens. Only such segments
  // signal q_ready (and only they make the MMA thread wait for it): an empty
  // unit's segment never waits on the MMA thread, so signalling for it could
  // complete two q_ready phases before the MMA thread observed the first.
  __device__ __forceinline__ bool begin_segment(int L, bool has_tokens) {
    // every softmax thread is done with the previous segment's row state
    // (its epilogue reads row_m) before it is reset here
    named_bar(kBarStage, C::kSoft);
    const int qs = nq % p.NQ;
    bool got = mbar_wait(sm.qfull(qs, p), (nq / p.NQ) & 1);
    got = __all_sync(0xffffffffu, got);
    if (!got) {
      fail();
      return false;
    }
    ++nq;
    Lseg = L;
    constexpr int TPR = C::kSoft / RN;  // threads per row
    constexpr int EPT = D / TPR;               // elements per thread
    static_assert(EPT % 16 == 0, "Q split granularity");
    const int tid = threadIdx.x;
    const int r = tid / TPR, part = tid % TPR;
    const bool valid = r < p.R;
    const uint32_t qrow = sm.qbuf(qs, p) + (uint32_t)(valid ? r : 0) * (uint32_t)(D * 2) + (uint32_t)part * EPT * 2u;
    uint4 raw[EPT / 8];
#pragma unroll
    for (int u = 0; u < EPT / 8; ++u) raw[u] = valid ? lds128(qrow + 16u * u) : make_uint4(0, 0, 0, 0);
    float cr = 0.f;
    if constexpr (FP8) {
      const bool qh = p.q_f16 != 0;  // FP16 queries (else BF16), widened exactly either way
      float amax = 0.f;
#pragma unroll
      for (int u = 0; u < EPT / 8; ++u) {
        const uint32_t w[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          amax = fmaxf(amax, fabsf(q_bits_to_f32(w[e] & 0xFFFFu, qh)));
          amax = fmaxf(amax, fabsf(q_bits_to_f32(w[e] >> 16, qh)));
        }
      }
#pragma unroll
      for (int off = 1; off < TPR; off <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
      // power-of-two row scale: the row's largest magnitude lands in [128, 256)
      int ex = 0;
      if (amax > 0.f) {
        const int e2 = (int)((__float_as_uint(amax) >> 23) & 0xFF) - 127;
        ex = max(-126, min(126, 7 - e2));
      }
      const float sc = __uint_as_float((uint32_t)(ex + 127) << 23);
      const float inv = __uint_as_float((uint32_t)(127 - ex) << 23);
      // four elements at a time: three e4m3 terms, one 32-bit word each (a
      // rolled loop: this runs once per segment, and short code misses the
      // instruction cache less often than it saves in issue slots)
#pragma unroll 1
      for (int g4 = 0; g4 < EPT / 4; ++g4) {
        // elements 4*g4 .. 4*g4+3: words 0-1 or 2-3 of 16-byte unit g4 / 2
        const uint32_t words[2] = {valid ? lds32(qrow + 8u * (uint32_t)g4) : 0u,
                                   valid ? lds32(qrow + 8u * (uint32_t)g4 + 4u) : 0u};
        float x[4], t0[4], t1[4], t2[4];
        x[0] = q_bits_to_f32(words[0] & 0xFFFFu, qh) * sc;
        x[1] = q_bits_to_f32(words[0] >> 16, qh) * sc;
        x[2] = q_bits_to_f32(words[1] & 0xFFFFu, qh) * sc;
        x[3] = q_bits_to_f32(words[1] >> 16, qh) * sc;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          t0[e] = e4m3_lead(x[e]);
          const float r1 = x[e] - t0[e];
          t1[e] = e4m3_lead(r1);
          t2[e] = r1 - t1[e];
        }
        const int dim0 = part * EPT + 4 * g4;
        const uint32_t off = (uint32_t)(dim0 / 128) * (RN * 128u) + (uint32_t)r * 128u +
                             (uint32_t)((((dim0 % 128) / 16) ^ (r & 7)) << 4) + (uint32_t)(dim0 % 16);
        sts32(q16() + off, pack_e4m3x4(t0[0], t0[1], t0[2], t0[3]));
        sts32(q16() + C::kQTermBytes + off, pack_e4m3x4(t1[0], t1[1], t1[2], t1[3]));
        sts32(q16() + 2 * C::kQTermBytes + off, pack_e4m3x4(t2[0], t2[1], t2[2], t2[3]));
      }
      cr = inv * p.sm_scale_log2 * (p.scale_mode == kScalePerTensor ? kscale : 1.f);
    } else {
#pragma unroll
      for (int u = 0; u < EPT / 8; ++u) {
        const int dim0 = part * EPT + 8 * u;
        sts128(q16() + (uint32_t)(dim0 / 64) * (RN * 128u) + (uint32_t)r * 128u +
                   (uint32_t)((((dim0 % 64) / 8) ^ (r & 7)) << 4),
               raw[u]);
      }
      cr = p.sm_scale_log2;
    }
    if (part == 0) {
      row_c()[r] = valid ? cr : 0.f;
      row_m()[r] = valid ? -INFINITY : INFINITY;  // rows past R never contribute
      row_pos()[r] = valid ? L - p.QL + r / p.G : 0;
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    named_bar(kBarStage, C::kSoft);
    __syncwarp();
    if (lane == 0) {
      if (has_tokens) mbar_arrive(bars.q_ready());
      mbar_arrive(sm.qempty(qs, p));
    }
    seg_k0 = k;
    return true;
  }

  // Every row's visible range covers the whole stage?
  __device__ __forceinline__ bool interior_stage(const StageView& h) const {
    return h.tbase >= h.t0 && h.tbase + TT <= h.t1 && (!p.causal || h.tbase + TT - 1 <= Lseg - p.QL) &&
           (p.window == 0 || h.tbase > Lseg - 1 - p.window);
  }
  __device__ __forceinline__ bool visible(const StageView& h, int pos) const {
    const int t = h.tbase + tok;
    if (t < h.t0 || t >= h.t1) return false;
    if (p.causal && t > pos) return false;
    if (p.window > 0 && t <= pos - p.window) return false;
    return true;
  }

  __device__ __forceinline__ void load_s(int buf, float (&s)[RH]) {
    uint32_t v[RH];
    tmem_ld_cols<RH>(tmem + lane_addr + C::kColS + (uint32_t)(buf * RN + wg * RH), v);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < RH; ++i) s[i] = __uint_as_float(v[i]);
  }

  // In place: y = s * c_r * ks - m_r (log2 units against the reference max),
  // -inf where masked; returns the largest y.
  __device__ __forceinline__ float scores(const StageView& h, bool interior, float ks, float (&y)[RH]) {
#pragma unroll
    for (int i = 0; i < RH; i += 4) {
      const float4 c4 = lds128f(row_c_u32(wg * RH + i));
      const float4 m4 = lds128f(row_m_u32(wg * RH + i));
      const float cc[4] = {c4.x, c4.y, c4.z, c4.w};
      const float mm[4] = {m4.x, m4.y, m4.z, m4.w};
      if (interior) {
#pragma unroll
        for (int j = 0; j < 4; ++j) y[i + j] = fmaf(VTOK ? y[i + j] * ks : y[i + j], cc[j], -mm[j]);
      } else {
        const int4 p4 = lds128i(row_pos_u32(wg * RH + i));
        const int pos[4] = {p4.x, p4.y, p4.z, p4.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float v = fmaf(VTOK ? y[i + j] * ks : y[i + j], cc[j], -mm[j]);
          y[i + j] = visible(h, pos[j]) ? v : -INFINITY;
        }
      }
    }
    return Max3Tree<RH>::run(y);  // the largest y
  }

  // Slow path (one warpgroup, for its own rows): raise the reference max of
  // rows whose stage maximum exceeds it by more than 2^8 and rescale their O
  // and L columns in tensor memory (after the previous PV has completed).
  // Leaves the stage's scores against the new reference in y.
  __device__ __forceinline__ bool raise_max(const StageView& h, bool interior, float ks, int buf, bool o_valid, float (&y)[RH]) {
    load_s(buf, y);
#pragma unroll
    for (int i = 0; i < RH; i += 4) {
      int pos[4] = {0, 0, 0, 0};
      if (!interior) {
        const int4 p4 = lds128i(row_pos_u32(wg * RH + i));
        pos[0] = p4.x;
        pos[1] = p4.y;
        pos[2] = p4.z;
        pos[3] = p4.w;
      }
      const float4 c4 = lds128f(row_c_u32(wg * RH + i));
      const float cc[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const bool vis = interior || visible(h, pos[j]);
        y[i + j] = vis ? (VTOK ? y[i + j] * ks : y[i + j]) * cc[j] : -INFINITY;
      }
    }
    {
      const float v = rowmax_transpose<RH>(y, lane);
      if (lane < RH) row_red()[quarter * 64 + wg * RH + lane] = v;
    }
    named_bar(kBarWg0 + wg, 128);
    if (threadIdx.x - 128 * wg < RH) {
      const int r = wg * RH + (threadIdx.x - 128 * wg);
      const float mold = row_m()[r];
      float smax = row_red()[r];
#pragma unroll
      for (int q = 1; q < 4; ++q) smax = fmaxf(smax, row_red()[q * 64 + r]);
      float alpha = 1.f;
      if (smax > mold + 8.f) {  // false for rows past R (reference +inf)
        alpha = (mold == -INFINITY) ? 0.f : ex2(mold - smax);
        row_m()[r] = smax;
      }
      row_alpha()[r] = alpha;
    }
    named_bar(kBarWg0 + wg, 128);
    bool any = false;
#pragma unroll
    for (int i = 0; i < RH; ++i) any |= row_alpha()[wg * RH + i] != 1.f;
    if (o_valid && any) {
      // O and L columns of this warpgroup's rows; the previous PV must be done
      if (!wait_pv(k - 1)) return false;
#pragma unroll 1
      for (int cblk = 0; cblk <= C::DCH; ++cblk) {  // DCH O^T blocks, then L^T
        const uint32_t col = (cblk < C::DCH ? C::kColO + (uint32_t)(cblk * RN) : C::kColL) + (uint32_t)(wg * RH);
        uint32_t v[RH];
        tmem_ld_cols<RH>(tmem + lane_addr + col, v);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < RH; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * row_alpha()[wg * RH + i]);
        tmem_st_cols<RH>(tmem + lane_addr + col, v);
      }
      tmem_wait_st();
    }
    load_s(buf, y);
    (void)scores(h, interior, ks, y);
    return true;
  }

  // This thread's FP8 V units (16 bytes each) of the stage: unit j is e =
  // threadIdx.x + 256 j, token e / (8 NCH), 128-byte chunk (e / 8) % NCH,
  // 16-byte column e % 8.
  static constexpr int kVUnits = TT * C::NCH * 8 / C::kSoft;
  __device__ __forceinline__ uint4 load_v_unit(uint32_t vst, int j) const {
    const int e = threadIdx.x + j * C::kSoft;
    const int t = e / (8 * C::NCH), cb = (e / 8) % C::NCH, cc = e % 8;
    return lds128(vst + (uint32_t)(cb * TT + t) * 128u + (uint32_t)((cc ^ (t & 7)) << 4));
  }
  // The unit as FP16 into the V^T operand over the stage's K and V bytes:
  // [D/64 chunks][TT][128 B]; tokens outside the stage's range become zeros
  // (poisoned slots never reach the MMA); per-token V scales (times 2^-4) are
  // folded in.
  __device__ __forceinline__ void store_v16_unit(uint32_t kst, uint32_t sst, const StageView& h, int j,
                                                 uint4 w) const {
    const int e = threadIdx.x + j * C::kSoft;
    const int t = e / (8 * C::NCH), cb = (e / 8) % C::NCH, cc = e % 8;
    const bool in = h.tbase + t >= h.t0 && h.tbase + t < h.t1;
    const int dim0 = cb * 128 + 16 * cc;
    const uint32_t dst =
        kst + (uint32_t)(dim0 / 64) * (TT * 128u) + (uint32_t)t * 128u + (uint32_t)((((dim0 % 64) / 8) ^ (t & 7)) << 4);
    uint4 lo, hi;
    lo.x = e4m3x2_to_f16x2(w.x & 0xFFFFu);
    lo.y = e4m3x2_to_f16x2(w.x >> 16);
    lo.z = e4m3x2_to_f16x2(w.y & 0xFFFFu);
    lo.w = e4m3x2_to_f16x2(w.y >> 16);
    hi.x = e4m3x2_to_f16x2(w.z & 0xFFFFu);
    hi.y = e4m3x2_to_f16x2(w.z >> 16);
    hi.z = e4m3x2_to_f16x2(w.w & 0xFFFFu);
    hi.w = e4m3x2_to_f16x2(w.w >> 16);
    if constexpr (VTOK) {
      float vs = in ? lds_f32(sst + 4u * (uint32_t)(TT + t)) : 0.f;
      if (in && !(fabsf(vs) <= 2048.f)) {
        flag_status(p, kStatusScaleRange);
        vs = 0.f;
      }
      const uint32_t s2 = pack_f16(vs * kVtokUnit, vs * kVtokUnit);
      lo.x = hmul2_bits(lo.x, s2);
      lo.y = hmul2_bits(lo.y, s2);
      lo.z = hmul2_bits(lo.z, s2);
      lo.w = hmul2_bits(lo.w, s2);
      hi.x = hmul2_bits(hi.x, s2);
      hi.y = hmul2_bits(hi.y, s2);
      hi.z = hmul2_bits(hi.z, s2);
      hi.w = hmul2_bits(hi.w, s2);
    }
    if (!in) lo = hi = make_uint4(0, 0, 0, 0);
    sts128(dst, lo);
    sts128(dst ^ 16u, hi);
  }
  // BF16 stage used in place: this thread zeroes its token's V row when the
  // token is outside the stage's range.
  __device__ __forceinline__ void clear_v_row(uint32_t vst, const StageView& h) const {
    const int t = h.tbase + tok;
    if (t >= h.t0 && t < h.t1) return;
#pragma unroll
    for (int cb = 0; cb < C::NCH; ++cb)
#pragma unroll
      for (int cc = 0; cc < 8; ++cc)
        sts128(vst + (uint32_t)(cb * TT + tok) * 128u + (uint32_t)(cc << 4), make_uint4(0, 0, 0, 0));
  }

  // One stage with tokens: scores -> P^T (and the FP16 V operand).
  __device__ __forceinline__ bool stage(const StageView& h, int s) {
    const int buf = k % C::SB;
    if (!mbar_wait(bars.s_full(buf), (k / C::SB) & 1)) {
      fail();
      return false;
    }
    tc_fence_after();
    const uint32_t kst = sm.stage(s, p);
    const uint32_t vst = kst + (uint32_t)TT * 128u * C::NCH;
    const uint32_t sst = kst + p.off_scale;
    const bool interior = interior_stage(h);
    const float ks = (VTOK && (h.tbase + tok >= h.t0 && h.tbase + tok < h.t1)) ? lds_f32(sst + 4u * tok) : 1.f;
    float y[RH];
    load_s(buf, y);
    const float mx = scores(h, interior, ks, y);
    // one vote per stage and warpgroup: some score of its rows above the
    // reference by more than 2^8? (The warpgroups own disjoint rows and O/L
    // columns, so they vote and rescale independently and may drift apart.)
    const bool o_valid = k > seg_k0;
    if (named_bar_or(kBarWg0 + wg, 128, mx > 8.f)) {
      if (!raise_max(h, interior, ks, buf, o_valid, y)) return false;
    }
    // S(k) is read: its buffer may take S(k + SB)
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bars.s_free(buf));
    // P^T row of this token (this warpgroup's RH rows), eight rows per 16-byte
    // store. FP8 caches: FP16 P in slot k % 3, last read by PV(k - 3). BF16
    // caches: hi = bf16(p), lo = bf16(p - hi) in the one buffer, last read by
    // PV(k - 1).
    if constexpr (FP8) {
      // FP16 V over the stage's K and V bytes, before waiting on the P slot.
      // Each FP16 chunk row of a token lies over that token's K bytes (which
      // S has consumed) or over its own FP8 V bytes, and all of a token's V
      // units are converted by lanes of one warp: every unit of the warp is
      // read before the warp writes any, which orders the in-place copy.
      uint4 wv[kVUnits];
#pragma unroll
      for (int j = 0; j < kVUnits; ++j) wv[j] = load_v_unit(vst, j);
      __syncwarp();
#pragma unroll
      for (int j = 0; j < kVUnits; ++j) store_v16_unit(kst, sst, h, j, wv[j]);
    } else if (!interior) {
      clear_v_row(vst, h);
    }
    if (k >= C::PB && !wait_pv(k - C::PB)) return false;
    const int slot0 = FP8 ? k % C::PB : 0;
    const uint32_t prow = pslot(slot0) + (uint32_t)tok * 128u;
#pragma unroll
    for (int u = 0; u < RH / 8; ++u) {
      uint32_t hw[4], lw[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float a = ex2(y[8 * u + 2 * i]), b = ex2(y[8 * u + 2 * i + 1]);  // ex2(-inf) = +0
        if constexpr (FP8) {
          hw[i] = pack_f16(a, b);
        } else {
          hw[i] = pack_bf16(a, b);
          lw[i] = pack_bf16(a - bf16_bits_to_f32(hw[i] & 0xFFFFu), b - bf16_bits_to_f32(hw[i] >> 16));
        }
      }
      const uint32_t off = (uint32_t)(((wg * (RH / 8) + u) ^ (tok & 7)) << 4);
      sts128(prow + off, make_uint4(hw[0], hw[1], hw[2], hw[3]));
      if constexpr (C::PT == 2) sts128(prow + TT * 128u + off, make_uint4(lw[0], lw[1], lw[2], lw[3]));
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(bars.p_full(buf));
      mbar_arrive(sm.empty(s, p));  // this warp is done with the stage
    }
    ++k;
    return true;
  }

  // Segment end: read O^T and L^T of this warpgroup's rows, write the BF16
  // output (a unit this CTA covers alone), a global partial or the cluster
  // partial; then the last-arriver or reducer bookkeeping.
  __device__ __forceinline__ void end_segment(const StageView& h, int slot, const MergeDesc& md) {
    const bool o_valid = k > seg_k0;
    if (o_valid && !wait_pv(k - 1)) return;
    const bool whole = (h.flags & kSegWhole) != 0;
    const bool cluster = p.merge == kMergeCluster;
    float* cp_o = reinterpret_cast<float*>(sm.base + p.off_cpart);
    float* cp_ml = cp_o + (size_t)p.Rpad * D;
    // Per row, the factor that turns O into the output (whole units:
    // sink-adjusted 1/L times the V scale) or into the partial (the per-token
    // V unit), into row_alpha; lane r of the warpgroup's first warp computes
    // row r's factor and writes a partial's (max, sum) pair.
    if (quarter == 0) {
      uint32_t v[RH];
      if (o_valid) {
        tmem_ld_cols<RH>(tmem + lane_addr + C::kColL + (uint32_t)(wg * RH), v);
        tmem_wait_ld();
      }
      float Lv = 0.f;
#pragma unroll
      for (int i = 0; i < RH; ++i) {
        // L^T rows are identical; lanes 0-15 of each quarter hold them (M = 64 layout)
        const float l = __shfl_sync(0xffffffffu, __uint_as_float(o_valid ? v[i] : 0u), lane & 15);
        if (lane == i) Lv = o_valid ? l : 0.f;
      }
      if (lane < RH) {
        const int r = wg * RH + lane;
        const float M = row_m()[r];
        float fr = VTOK ? 1.f / kVtokUnit : 1.f;
        if (whole) {
          float L = Lv, a = 1.f;
          if (p.has_sinks && r < p.R) {
            const float s2 = __ldg(p.sinks + h.g * p.G + r % p.G) * kLog2e;
            const float M2 = fmaxf(M, s2);
            a = (M == -INFINITY) ? 0.f : ex2(M - M2);
            L = fmaf(L, a, ex2(s2 - M2));
          }
          fr = (L > 0.f) ? a * ((1.f / L) * vscale) : 0.f;
        } else if (r < p.R) {
          const float2 ml = make_float2(M, Lv);
          if (cluster)
            *reinterpret_cast<float2*>(cp_ml + 2 * r) = ml;
          else
            *reinterpret_cast<float2*>(p.part_ml + ((size_t)slot * p.Rpad + r) * 2) = ml;
        }
        row_alpha()[r] = fr;
      }
    }
    named_bar(kBarWg0 + wg, 128);
    // O * f through shared memory (the P slots, idle once the last PV is
    // done: [RN rows][D] f32), then every softmax thread writes 16-byte
    // pieces of whole rows: fewer, wider stores than one float per row.
    const uint32_t stg = sm.base_u32 + p.off_p16;
#pragma unroll 1
    for (int cblk = 0; cblk < C::DCH; ++cblk) {
      const int d = cblk * 128 + tok;  // lane quarter q, lane l -> dim 32q + l of this block
      // 16 columns at a time keeps the live registers low
#pragma unroll
      for (int hh = 0; hh < RH / 16; ++hh) {
        uint32_t v[16];
        if (o_valid) {
          tmem_ld16(tmem + lane_addr + C::kColO + (uint32_t)(cblk * RN + wg * RH + 16 * hh), v);
          tmem_wait_ld();
        }
#pragma unroll
        for (int i = 0; i < 16; i += 4) {
          const float4 f4 = lds128f(row_alpha_u32(wg * RH + 16 * hh + i));
          const float fq[4] = {f4.x, f4.y, f4.z, f4.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float o = (o_valid ? __uint_as_float(v[i + j]) : 0.f) * fq[j];
            asm volatile("st.shared.f32 [%0], %1;" ::"r"(stg + 4u * (uint32_t)((wg * RH + 16 * hh + i + j) * D + d)),
                         "f"(o)
                         : "memory");
          }
        }
      }
    }
    named_bar(kBarStage, C::kSoft);
    {
      const int E = p.R * (D / 4);  // float4 pieces of the R rows
      for (int e = threadIdx.x; e < E; e += C::kSoft) {
        const int r = e / (D / 4), d = (e % (D / 4)) * 4;
        const float4 o = lds128f(stg + 4u * (uint32_t)(r * D + d));
        if (whole) {
          const int qi = r / p.G, head = h.g * p.G + r % p.G;
          uint2 st;
          st.x = pack_out(o.x, o.y, p.q_f16 != 0);
          st.y = pack_out(o.z, o.w, p.q_f16 != 0);
          *reinterpret_cast<uint2*>(p.out + ((size_t)(h.b * p.QL + qi) * p.Hq + head) * D + d) = st;
        } else if (cluster) {
          *reinterpret_cast<float4*>(cp_o + (size_t)r * D + d) = o;
        } else {
          *reinterpret_cast<float4*>(p.part_o + ((size_t)slot * p.Rpad + r) * D + d) = o;
        }
      }
    }
    // O and L are read; the next segment's first PV may overwrite them
    tc_fence_before();
    if (whole || cluster) return;
    if (p.merge == kMergeReducer) {
      if (threadIdx.x == 0 && slot == md.s0) p.unit_desc[h.unit] = make_int4(md.nseg, md.s0, md.sbase, md.sstride);
    } else if (p.merge == kMergeLastArriver) {
      __threadfence();
      named_bar(1, C::kSoft);
      if (threadIdx.x == 0) la_arrive(p, sm, h.b, h.g, h.unit, md);
      named_bar(1, C::kSoft);
      la_run_queue<D>(p, sm, per_tensor_vscale(p), C::kSoft);
    }
  }

  __device__ __forceinline__ void run() {
    StageView h;
    while (ok) {
      const int s = n % p.NS;
      bool got = mbar_wait(sm.full(s, p), (n / p.NS) & 1);
      got = __all_sync(0xffffffffu, got);
      if (!got) {
        fail();
        break;
      }
      const uint32_t ha = sm.hdr_u32(s, p);
      const int4 h0 = lds128i(ha);
      if (h0.x & kEnd) break;
      const int4 h1 = lds128i(ha + 16);
      h.flags = h0.x;
      h.tbase = h0.y;
      h.t0 = h0.z;
      h.t1 = h0.w;
      h.L = h1.x;
      h.unit = h1.y;
      h.b = h1.z;
      h.g = h1.w;
      h.m0 = h.m1 = h.m2 = h.m3 = 0u;
      int slot = 0;
      MergeDesc md{1, 0, 0, 0};
      if (h.flags & kSegLast) {
        const int4 h3 = lds128i(ha + 48);
        const int sstride = lds128i(ha + 64).x;
        slot = h3.x;
        md = MergeDesc{h3.y, h3.z, h3.w, sstride};
      }
      if ((h.flags & kSegFirst) && !begin_segment(h.L, h.t1 > h.t0)) break;
      if (h.t1 > h.t0) {
        if (!stage(h, s)) break;
      } else {
        __syncwarp();
        if (lane == 0) mbar_arrive(sm.empty(s, p));
      }
      if (h.flags & kSegLast) end_segment(h, slot, md);
      ++n;
    }
  }
};

// The MMA-issuing thread (lane 0 of the warp after the producer).
template <bool FP8, int D, bool VTOK, int RH, int NWG>
struct MtpIssuer {
  using C = MtpCfg<FP8, D, VTOK, RH, NWG>;
  static constexpr int TT = C::TT;
  static constexpr int RN = C::RN;
  const PaParams& p;
  Smem sm;
  MtpBars bars;
  uint32_t tmem;
  uint64_t dq, dones, dp0;
  bool ok = true;

  __device__ __forceinline__ MtpIssuer(const PaParams& p_, Smem s, uint32_t tm) : p(p_), sm(s), tmem(tm) {
    bars.base = sm.base_u32 + p.off_ubar;
    dq = umma_sdesc(sm.base_u32 + p.off_q16, 16, 1024);
    dp0 = umma_sdesc(sm.base_u32 + p.off_p16, TT * 128u, 1024);
    // the ones operand: 2 KiB of 1.0 read as [64 x 16] without swizzle (any
    // core-matrix strides that stay inside the buffer read the same values)
    dones = umma_sdesc_noswz(sm.base_u32 + p.off_p16 + (uint32_t)C::NP * TT * 128u, 128, 256);
  }
  __device__ __forceinline__ static uint64_t dadd(uint64_t d, uint32_t byte_off) { return d + (uint64_t)(byte_off >> 4); }

  __device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity) {
    if (mbar_wait(bar, parity)) return true;
    ok = false;
    flag_status(p, kStatusTimeout);
    return false;
  }

  // S^T(k) = K . Q^T into buffer k % SB
  __device__ __forceinline__ void issue_s(int buf, uint32_t kst) {
    const uint64_t dk = umma_sdesc(kst, 16, 1024);
    const uint32_t d = tmem + C::kColS + (uint32_t)(buf * RN);
    if constexpr (FP8) {
      // three Q terms accumulate into one S; 32 e4m3 values per k-step
#pragma unroll
      for (int t = 0; t < 3; ++t)
#pragma unroll
        for (int j = 0; j < D / 32; ++j)
          umma_f8(d, dadd(dk, (uint32_t)(j / 4) * (TT * 128u) + (uint32_t)(j % 4) * 32u),
                  dadd(dq, (uint32_t)t * C::kQTermBytes + (uint32_t)(j / 4) * (RN * 128u) + (uint32_t)(j % 4) * 32u),
                  C::kIdS, (t > 0 || j > 0) ? 1u : 0u);
    } else {
#pragma unroll
      for (int j = 0; j < D / 16; ++j)
        umma_f16(d, dadd(dk, (uint32_t)(j / 4) * (TT * 128u) + (uint32_t)(j % 4) * 32u),
                 dadd(dq, (uint32_t)(j / 4) * (RN * 128u) + (uint32_t)(j % 4) * 32u), C::kIdS, j > 0 ? 1u : 0u);
    }
    umma_commit(bars.s_full(buf));
  }

  // O^T += V^T . P^T(kk), L^T += 1 . P^T(kk) (P(kk) is ready); then release
  // stage s.
  __device__ __forceinline__ void issue_pv(int kk, int s, bool acc) {
    tc_fence_after();
    const uint32_t kst = sm.stage(s, p);
    // V^T: FP8 caches -> FP16 copy over the stage's K and V bytes; BF16 -> the V bytes
    const uint32_t vbase = FP8 ? kst : kst + (uint32_t)TT * 128u * C::NCH;
    const uint64_t dv = umma_sdesc(vbase, TT * 128u, 1024);
#pragma unroll
    for (int t = 0; t < C::PT; ++t) {
      const uint64_t dp = dadd(dp0, (uint32_t)((FP8 ? kk % C::PB : 0) + t) * (TT * 128u));
      const bool a0 = acc || t > 0;
#pragma unroll
      for (int cblk = 0; cblk < C::DCH; ++cblk)
#pragma unroll
        for (int j = 0; j < TT / 16; ++j)
          umma_f16(tmem + C::kColO + (uint32_t)(cblk * RN),
                   dadd(dv, (uint32_t)cblk * (2u * TT * 128u) + (uint32_t)j * 2048u), dadd(dp, (uint32_t)j * 2048u),
                   C::kIdPV, (a0 || j > 0) ? 1u : 0u);
#pragma unroll
      for (int j = 0; j < TT / 16; ++j)
        umma_f16(tmem + C::kColL, dones, dadd(dp, (uint32_t)j * 2048u), C::kIdL, (a0 || j > 0) ? 1u : 0u);
    }
    umma_commit(bars.pv_done(kk % 3));
    umma_commit(sm.empty(s, p));
  }

  // Phase wait that gives up after a short suspend (~500 ns).
  __device__ __forceinline__ static bool wait_hint(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(500u)
        : "memory");
    return ok != 0;
  }

  // Non-blocking phase test of an mbarrier.
  __device__ __forceinline__ static bool ready(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
  }

  // Event loop: S(k) is issued as soon as stage k's bytes, the segment's Q
  // operand and S buffer k % SB are ready; PV(j) as soon as P(j) is, in order.
  // The two streams interleave freely, so a stage is released right after
  // its PV and never waits for the next stage's data.
  __device__ __forceinline__ void run() {
    int n = 0;          // next ring stage to examine
    int ks = 0;         // S issued so far
    int kp = 0;         // PV issued so far
    int qn = 0;         // segments whose Q operand was awaited
    bool seg_acc = false;
    bool done = false;  // end marker seen
    bool hdr_ok = false, need_q = false;  // stage n's header read (and its Q wait pending)
    int hflags = 0;
    bool htok = false;
    // pending PVs in issue order (at most SB: S runs at most SB stages ahead
    // of the softmax): ring stage and whether O accumulates
    int pv_st0 = 0, pv_st1 = 0, pv_st2 = 0;
    bool pv_ac0 = false, pv_ac1 = false, pv_ac2 = false;
    static_assert(C::SB <= 3, "pending-PV queue depth");
    unsigned long long idle_since = 0;
    while (ok) {
      bool progress = false;
      // PV(kp) as soon as P(kp) is ready
      if (kp < ks && ready(bars.p_full(kp % C::SB), (kp / C::SB) & 1)) {
        issue_pv(kp, pv_st0, pv_ac0);
        pv_st0 = pv_st1;
        pv_ac0 = pv_ac1;
        pv_st1 = pv_st2;
        pv_ac1 = pv_ac2;
        ++kp;
        progress = true;
      } else if (!done) {
        const int s = n % p.NS;
        if (!hdr_ok && ready(sm.full(s, p), (n / p.NS) & 1)) {
          const int4 h0 = lds128i(sm.hdr_u32(s, p));
          hdr_ok = true;
          hflags = h0.x;
          htok = h0.w > h0.z;
          need_q = (hflags & kSegFirst) != 0 && htok;  // empty segments signal no q_ready
          if (hflags & kEnd) done = true;
          progress = true;
        }
        if (hdr_ok && !done) {
          if (need_q && ready(bars.q_ready(), qn & 1)) {
            need_q = false;
            ++qn;
            seg_acc = false;
            progress = true;
          }
          if (!need_q) {
            if (!htok) {
              mbar_arrive(sm.empty(s, p));  // no MMA reads this stage
              hdr_ok = false;
              ++n;
              progress = true;
            } else if (ks - kp < C::SB && (ks < C::SB || ready(bars.s_free(ks % C::SB), (ks / C::SB - 1) & 1))) {
              tc_fence_after();
              issue_s(ks % C::SB, sm.stage(s, p));
              const int q = ks - kp;  // queue position of PV(ks)
              if (q == 0) {
                pv_st0 = s;
                pv_ac0 = seg_acc;
              } else if (q == 1) {
                pv_st1 = s;
                pv_ac1 = seg_acc;
              } else {
                pv_st2 = s;
                pv_ac2 = seg_acc;
              }
              seg_acc = true;
              ++ks;
              hdr_ok = false;
              ++n;
              progress = true;
            }
          }
        }
      }
      if (done && kp == ks) break;
      if (progress) {
        idle_since = 0;
      } else {
        // Nothing ready: sleep (at most ~0.5 us) on the event most likely to
        // come next instead of spinning on the issue slots the softmax warps
        // of this sub-partition need.
        if (kp < ks)
          (void)wait_hint(bars.p_full(kp % C::SB), (kp / C::SB) & 1);
        else if (!done && !hdr_ok)
          (void)wait_hint(sm.full(n % p.NS, p), (n / p.NS) & 1);
        else if (!done && need_q)
          (void)wait_hint(bars.q_ready(), qn & 1);
        else if (!done && ks >= C::SB)
          (void)wait_hint(bars.s_free(ks % C::SB), (ks / C::SB - 1) & 1);
        const unsigned long long t = global_timer();
        if (idle_since == 0) {
          idle_since = t;
        } else if (t - idle_since > kWaitLimitNs) {
          ok = false;
          flag_status(p, kStatusTimeout);
        }
      }
    }
    // every issued MMA completes before the CTA frees tensor memory
    umma_commit(bars.drained());
    if (!mbar_wait_spin(bars.drained(), 0)) flag_status(p, kStatusTimeout);
  }
};

// Softmax warps 0 .. 4 NWG - 1, then the producer warp and the MMA warp.
template <bool FP8, int D, bool VTOK, int RH, int NWG>
__global__ void __launch_bounds__(MtpCfg<FP8, D, VTOK, RH, NWG>::kThreads, 1)
    pa_mtp_kernel(const __grid_constant__ PaParams p, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV) {
  using Cfg = MtpCfg<FP8, D, VTOK, RH, NWG>;
  extern __shared__ uint8_t smem_raw[];
  Smem sm;
  {
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t aligned = (raw + 1023u) & ~1023u;
    sm.base = smem_raw + (aligned - raw);
    sm.base_u32 = aligned;
  }
  const int warp = threadIdx.x >> 5;
  if (warp == 0) prefetch_params(p);
  const uint32_t bar0 = sm.base_u32 + p.off_ubar;
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.NS; ++s) {
      mbar_init(sm.full(s, p), 1);
      mbar_init(sm.empty(s, p), Cfg::kSoftWarps + 1);  // softmax warps + the MMA commit (or the MMA thread)
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(sm.qfull(i, p), 1);
      mbar_init(sm.qempty(i, p), Cfg::kSoftWarps);
    }
    for (int i = 0; i < 3; ++i) {
      mbar_init(bar0 + 8u * i, 1);                      // s_full: MMA commit
      mbar_init(bar0 + 24u + 8u * i, Cfg::kSoftWarps);  // s_free: softmax warps
      mbar_init(bar0 + 48u + 8u * i, Cfg::kSoftWarps);  // p_full: softmax warps
      mbar_init(bar0 + 72u + 8u * i, 1);                // pv_done: MMA commit
    }
    mbar_init(bar0 + 96u, Cfg::kSoftWarps);  // q_ready
    mbar_init(bar0 + 104u, 1);               // drained
    for (int i = 0; i < 16; ++i) sm.misc(p)[i] = 0;
    fence_barrier_init();
  }
  // the ones operand of the row sums (64 x 16 elements of 1.0, layout-free)
  {
    const uint32_t one2 = FP8 ? 0x3C003C00u : 0x3F803F80u;
    const uint32_t ones = sm.base_u32 + p.off_p16 + (uint32_t)Cfg::NP * kMtpTT * 128u;
    for (uint32_t o = threadIdx.x * 16u; o < 2048u; o += Cfg::kThreads * 16u) sts128(ones + o, make_uint4(one2, one2, one2, one2));
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(sm.base_u32 + p.off_tslot),
                 "r"(Cfg::kCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sm.base + p.off_tslot);
  constexpr int ELT = FP8 ? 1 : 2;
  constexpr int NCH = D * ELT / 128;
  if (warp == Cfg::kProducerWarp) {
    Producer<ELT, NCH> prod(p, &tmK, &tmV, sm);
    prod.run();
    if (p.merge == kMergeCluster) {
      cluster_sync_all();
      cluster_sync_all();
    }
  } else if (warp == Cfg::kMmaWarp) {
    if ((threadIdx.x & 31) == 0) {
      MtpIssuer<FP8, D, VTOK, RH, NWG> mma(p, sm, tmem);
      mma.run();
    }
    __syncwarp();
    if (p.merge == kMergeCluster) {
      cluster_sync_all();
      cluster_sync_all();
    }
  } else {
    MtpSoftmax<FP8, D, VTOK, RH, NWG> cons(p, sm, tmem);
    cons.run();
    if (p.merge == kMergeCluster) {
      cluster_sync_all();
      cluster_merge_unit<D>(p, sm, per_tensor_vscale(p), blockIdx.x / p.P, threadIdx.x, Cfg::kSoft);
      cluster_sync_all();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(Cfg::kCols) : "memory");
  }
}

}  // namespace dev
}  // namespace pa
