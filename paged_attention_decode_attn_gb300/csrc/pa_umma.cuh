// Tensor-memory (tcgen05) consumer for query-row groups of 17..64 rows per KV
// head (MTP verify rows x GQA), dense paged decode on sm_103a.
//
// The producer warp, the stage ring, the Q ring, the schedules and the
// partial merges are those of the tile kernel (pa_tile.cuh). A stage is
// consumed with tcgen05.mma chains issued by one thread, accumulators in
// tensor memory:
//
//   S^T[TT x N] = K[TT x D] . Q^T     (M = the stage's tokens; N = 64 rows)
//   O[M x D]   += P[M x TT] . V        (A = P^T and B = V both MN-major)
//   L[M x 16]  += P . ones             (the row sums, from the tensor cores)
//
// One thread holds one token's row of S^T (warps w and w + 4 share TMEM lane
// quarter w and split its 64 row scores), applies scale and masks, and writes
// its token's row of P^T. The softmax keeps a lazy reference max per row: P is
// taken against it, and only a score more than 2^8 above it (always on a
// segment's first stage, rarely later) sends the CTA through a slow path that
// reduces the stage's row maxima across threads and rescales O and L in TMEM.
// The row owners (M = 64: lane l < 16 of warp q holds row 16q + l) read O and
// L at the segment end.
//
// Operands (128-byte swizzle, 128-byte chunks):
//  * BF16 caches: the stage is read in place; Q and P BF16 (kind::f16).
//  * FP8 caches, head_dim 128, per-tensor scales: the stage is read in place by
//    kind::f8f6f4 MMAs; Q and P enter as two-term e4m3 sums hi + lo, stacked
//    as 128 rows, so S^T has 128 columns (hi and lo halves added per row) and
//    O and L 128 lanes (halves added at the segment end).
//  * other FP8 shapes: K and V converted exactly to FP16 in their row layout
//    (V stays an MN-major operand, no transpose); Q in FP16 under an exact
//    power-of-two row scale, P in FP16 below 2^8.
//
// Sources of the method: the tile kernel's pages (split-KV partials, scale
// before mask, per-token scales folded into P, MTP rows); the tensor-memory
// layout, the operand splits and the ordering of the MMA chains are this
// implementation's.
#pragma once

#include <cuda_fp8.h>

#include "pa_tile.cuh"

namespace pa {
namespace dev {

// ------------------------------------------------------------ tcgen05 helpers
// Shared-memory matrix descriptor, 128-byte swizzle.
__device__ __forceinline__ uint64_t umma_sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version
  d |= (uint64_t)2 << 61;  // 128-byte swizzle
  return d;
}
// Instruction descriptor, kind::f16: FP32 accumulate, A and B both FP16 or
// both BF16, each K-major or MN-major.
__host__ __device__ constexpr uint32_t umma_idesc_ab(bool bf16, int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | ((a_mn_major ? 1u : 0u) << 15) |
         ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Four floats -> four e4m3 bytes (first value in the lowest byte), RN, saturating.
__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return lo | (hi << 16);
}
// Leading term of a two-term e4m3 split: x rounded to nearest-even at 4
// significant bits, which e4m3 holds exactly for 2^-6 <= |x| <= 448; 0 below
// 2^-6 (the trailing term x - lead then carries all of x).
__device__ __forceinline__ float e4m3_lead(float x) {
  const float ax = fabsf(x);
  if (ax < 0.015625f) return 0.f;
  uint32_t u = __float_as_uint(ax);
  u = (u + 0x7FFFFu + ((u >> 20) & 1u)) & 0xFFF00000u;
  return copysignf(__uint_as_float(u), x);
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]),
        "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
        "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
      "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
      "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// Bounded spin on an MMA commit barrier (no suspend hint: the commit's
// arrival is polled directly).
__device__ __forceinline__ bool mbar_wait_spin(uint32_t bar, uint32_t parity) {
  uint32_t done = 0;
  const unsigned long long t0 = global_timer();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i) {
      asm volatile(
          "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
          : "=r"(done)
          : "r"(bar), "r"(parity)
          : "memory");
      if (done) return true;
    }
    if (global_timer() - t0 > kWaitLimitNs) return false;
  }
}
// Named barrier that also ORs a predicate over the participating threads.
__device__ __forceinline__ bool named_bar_or(int id, int nthr, bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred pi, po;\n setp.ne.u32 pi, %2, 0;\n barrier.cta.red.or.pred po, %1, %3, pi;\n"
      " selp.u32 %0, 1, 0, po;\n}\n"
      : "=r"(r)
      : "r"(id), "r"((uint32_t)v), "r"(nthr)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

constexpr int kUmmaRows = 64;      // query rows of the MMA block (N of S^T, M of O)
constexpr int kUmmaThreads = 256;  // eight consumer warps: warps w and w + 4 share TMEM lane quarter w
constexpr int kHalfRows = 32;      // score rows per thread (warps 0-3: rows 0-31, warps 4-7: rows 32-63)
constexpr uint32_t kUmmaOCol = 64;  // TMEM columns: S^T [0, 64), O [64, 64 + D), L [64 + D, +16)

template <bool FP8, int D, bool VTOK>
struct UmmaConsumer {
  static constexpr int ELT = FP8 ? 1 : 2;
  static constexpr int NCH = D * ELT / 128;         // 128-byte blocks per token row of a stage
  static constexpr int TT = 32768 / (2 * D * ELT);  // tokens per stage (M of S^T)
  // FP8 at head_dim 128 with per-tensor scales: FP8 MMAs (kind::f8f6f4) read
  // K and V from the stage itself; Q and P enter as two-term FP8 sums
  // (hi + lo), stacked as 128 rows. Otherwise FP8 stages are converted to
  // FP16 operands (CONV): with per-token scales P is multiplied by the V
  // scale (~amax/448), which would put most of P * v_scale in e4m3's
  // subnormal range, where the two-term sum loses its precision.
  static constexpr bool F8 = FP8 && D == 128 && !VTOK;
  static constexpr bool CONV = FP8 && !F8;
  static constexpr int SN = F8 ? 128 : kUmmaRows;  // N of S^T
  static constexpr int OM = F8 ? 128 : kUmmaRows;  // M of O and L
  static constexpr uint32_t kOCol = F8 ? 128u : kUmmaOCol;
  static constexpr uint32_t kLCol = kOCol + D;  // row sums, 16 equal columns
  static constexpr uint32_t kTmemCols = (kLCol + 16) <= 256 ? 256u : 512u;
  static_assert(TT == 64 || TT == 128, "stage tokens");
  // S^T = K Q^T: M = TT tokens, N = SN rows, A = K (K-major), B = Q (K-major)
  static constexpr uint32_t kIdescS = umma_idesc_ab(!FP8, TT, SN, false, false);
  // O += P V: M = OM rows, N = D, A = P^T (MN-major), B = V (MN-major)
  static constexpr uint32_t kIdescPV = umma_idesc_ab(!FP8, OM, D, true, true);
  // L += P 1: N = 16, B = ones (K-major)
  static constexpr uint32_t kIdescL = umma_idesc_ab(!FP8, OM, 16, true, false);

  const PaParams& p;
  Smem sm;
  int warp, lane;
  int r;          // O row owned by this thread (M = 64 layout: lane < 16 of warp w -> row 16w + lane)
  int olane_row;  // row whose O lane this thread reads (F8: lane 32q + l -> row (32q + l) % 64)
  bool row_own;   // r < R
  int tok;        // S^T row (stage token) held by this thread, -1 if none
  int half;       // which 32 of the 64 rows this thread's softmax covers
  uint32_t tmem = 0, lane_base = 0;
  float kscale = 1.f, vscale = 1.f;
  bool o_valid = false, pv_pending = false;
  int nq = 0;
  uint32_t ph_s = 0, ph_o = 0;
  int pend_stage = -1;  // stage read in place by the outstanding PV (BF16, FP8 MMAs), handed back when it completes
  bool ok = true;
  // operand descriptors (built once) and barrier addresses
  uint64_t dq = 0, dpt = 0, dpu = 0, dones = 0, dk16 = 0, dv16 = 0;
  uint32_t sbar_addr = 0, obar_addr = 0;

  __device__ UmmaConsumer(const PaParams& p_, Smem s) : p(p_), sm(s) {
    warp = threadIdx.x >> 5;
    lane = threadIdx.x & 31;
    const int quarter = warp & 3;
    half = warp >> 2;
    if constexpr (F8) {
      // O lanes 0..63 hold the rows' hi parts, 64..127 the lo parts
      olane_row = (32 * quarter + lane) & 63;
      r = olane_row;
      row_own = half == 0 && quarter < 2 && r < p.R;
    } else {
      r = 16 * quarter + lane;
      olane_row = r;
      row_own = half == 0 && lane < 16 && r < p.R;
    }
    // M = 128: token 32q + lane; M = 64: token 16q + lane for lane < 16
    tok = TT == 128 ? 32 * quarter + lane : (lane < 16 ? 16 * quarter + lane : -1);
    lane_base = (uint32_t)(32 * quarter) << 16;
    if (FP8 && p.scale_mode == kScalePerTensor) kscale = __ldg(p.k_scale);
    vscale = per_tensor_vscale(p);
  }

  __device__ __forceinline__ uint32_t q16() const { return sm.base_u32 + p.off_q16; }
  __device__ __forceinline__ uint32_t pt16() const { return sm.base_u32 + p.off_p16; }
  // unscaled P^T for the row sums when per-token V scales are folded into P
  __device__ __forceinline__ uint32_t pu16() const { return sm.base_u32 + p.off_p16 + TT * 128; }
  __device__ __forceinline__ uint32_t ones16() const { return sm.base_u32 + p.off_p16 + (VTOK ? 2 : 1) * TT * 128; }
  __device__ __forceinline__ uint32_t sbar() const { return sm.base_u32 + p.off_ubar; }
  __device__ __forceinline__ uint32_t obar() const { return sm.base_u32 + p.off_ubar + 8; }
  // per-row state in shared memory (64 entries each)
  __device__ __forceinline__ float* row_c() const { return reinterpret_cast<float*>(sm.base + p.off_rows); }
  __device__ __forceinline__ float* row_m() const { return row_c() + kUmmaRows; }
  __device__ __forceinline__ int* row_pos() const { return reinterpret_cast<int*>(row_c() + 2 * kUmmaRows); }
  __device__ __forceinline__ float* row_alpha() const { return row_c() + 3 * kUmmaRows; }
  __device__ __forceinline__ float* row_smax() const { return row_c() + 4 * kUmmaRows; }  // [4 warps][64]
  __device__ __forceinline__ int* flags() const { return reinterpret_cast<int*>(row_c() + 8 * kUmmaRows); }
  // 16-byte unit u of row `row` in 64-element chunk c of a [chunks][rows][128 B] swizzled operand
  __device__ __forceinline__ static uint32_t swz_unit(uint32_t base, int c, int rows, int row, int u) {
    return base + (uint32_t)c * (uint32_t)rows * 128u + (uint32_t)row * 128u + (uint32_t)((u ^ (row & 7)) << 4);
  }

  __device__ void fail() {
    ok = false;
    if (lane == 0) {
      flag_status(p, kStatusTimeout);
      sm.misc(p)[0] |= 1;
    }
  }

  __device__ void setup() {
    for (uint32_t o = threadIdx.x * 16u; o < (uint32_t)(kUmmaRows * D * 2); o += kUmmaThreads * 16u)
      sts128(q16() + o, make_uint4(0, 0, 0, 0));
    // ones operand (16 x TT, K-major; every element 1.0)
    const uint32_t one2 = F8 ? 0x38383838u : (FP8 ? 0x3C003C00u : 0x3F803F80u);
    for (uint32_t o = threadIdx.x * 16u; o < (uint32_t)(16 * TT * (F8 ? 1 : 2)); o += kUmmaThreads * 16u)
      sts128(ones16() + o, make_uint4(one2, one2, one2, one2));
    if (warp == 0) {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(sm.base_u32 + p.off_tslot),
                   "r"(kTmemCols)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    named_bar(1, kUmmaThreads);
    tc_fence_after();
    tmem = *reinterpret_cast<volatile uint32_t*>(sm.base + p.off_tslot);
    dq = umma_sdesc(q16(), 16, 1024);
    dpt = umma_sdesc(pt16(), TT * 128u, 1024);
    dpu = umma_sdesc(pu16(), TT * 128u, 1024);
    dones = umma_sdesc(ones16(), 16, 1024);
    dk16 = umma_sdesc(sm.base_u32 + p.off_k16, 16, 1024);
    dv16 = umma_sdesc(sm.base_u32 + p.off_v16, TT * 128u, 1024);
    sbar_addr = sbar();
    obar_addr = obar();
  }

  __device__ void teardown() {
    if (pv_pending) wait_pv();
    tc_fence_before();
    named_bar(1, kUmmaThreads);
    if (warp == 0)
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }

  __device__ void wait_pv() {
    if (!mbar_wait_spin(obar(), ph_o)) fail();
    ph_o ^= 1u;
    pv_pending = false;
    tc_fence_after();
    if (pend_stage >= 0) {
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.empty(pend_stage, p));
      pend_stage = -1;
    }
  }

  // Query rows into the Q operand, per-row score scale and position, reset
  // of the reference max (+inf for rows past R, so they never contribute).
  __device__ bool begin_segment(int L) {
    const int qs = nq % p.NQ;
    bool got = mbar_wait(sm.qfull(qs, p), (nq / p.NQ) & 1);
    got = __all_sync(0xffffffffu, got);
    if (!got) return false;
    ++nq;
    if (threadIdx.x < kUmmaRows) {
      const int rr = threadIdx.x;
      float c = 0.f;
      if (rr < p.R) {
        const uint32_t qrow = sm.qbuf(qs, p) + (uint32_t)rr * (uint32_t)(D * 2);
        if constexpr (F8) {
          // power-of-two row scale to a max in [128, 256), then q = hi + lo
          // in e4m3 (rows rr and 64 + rr of the Q operand)
          float amax = 0.f;
          for (int u = 0; u < D / 8; ++u) {
            const uint4 w = lds128(qrow + 16u * u);
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              amax = fmaxf(amax, fabsf(bf16_bits_to_f32(ws[e] & 0xFFFFu)));
              amax = fmaxf(amax, fabsf(bf16_bits_to_f32(ws[e] >> 16)));
            }
          }
          int ex = 0;
          if (amax > 0.f) {
            const int e2 = (int)((__float_as_uint(amax) >> 23) & 0xFF) - 127;
            ex = max(-126, min(126, 7 - e2));
          }
          const float sc = __uint_as_float((uint32_t)(ex + 127) << 23);
          const float inv = __uint_as_float((uint32_t)(127 - ex) << 23);
          for (int u = 0; u < D / 16; ++u) {  // 16 values = one 16-byte unit of a row
            const uint4 w0 = lds128(qrow + 32u * u), w1 = lds128(qrow + 32u * u + 16u);
            const uint32_t ws[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
            float hv[16], lv[16];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float a = bf16_bits_to_f32(ws[e] & 0xFFFFu) * sc, b = bf16_bits_to_f32(ws[e] >> 16) * sc;
              hv[2 * e] = e4m3_lead(a);
              hv[2 * e + 1] = e4m3_lead(b);
              lv[2 * e] = a - hv[2 * e];
              lv[2 * e + 1] = b - hv[2 * e + 1];
            }
            const uint4 ho = make_uint4(pack_e4m3x4(hv[0], hv[1], hv[2], hv[3]), pack_e4m3x4(hv[4], hv[5], hv[6], hv[7]),
                                        pack_e4m3x4(hv[8], hv[9], hv[10], hv[11]),
                                        pack_e4m3x4(hv[12], hv[13], hv[14], hv[15]));
            const uint4 lo = make_uint4(pack_e4m3x4(lv[0], lv[1], lv[2], lv[3]), pack_e4m3x4(lv[4], lv[5], lv[6], lv[7]),
                                        pack_e4m3x4(lv[8], lv[9], lv[10], lv[11]),
                                        pack_e4m3x4(lv[12], lv[13], lv[14], lv[15]));
            sts128(swz_unit(q16(), 0, 128, rr, u), ho);
            sts128(swz_unit(q16(), 0, 128, 64 + rr, u), lo);
          }
          c = inv * p.sm_scale_log2 * (p.scale_mode == kScalePerTensor ? kscale : 1.f);
        } else if constexpr (FP8) {
          float amax = 0.f;
          for (int u = 0; u < D / 8; ++u) {
            const uint4 w = lds128(qrow + 16u * u);
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              amax = fmaxf(amax, fabsf(bf16_bits_to_f32(ws[e] & 0xFFFFu)));
              amax = fmaxf(amax, fabsf(bf16_bits_to_f32(ws[e] >> 16)));
            }
          }
          int ex = 0;
          if (amax > 0.f) {
            const int e2 = (int)((__float_as_uint(amax) >> 23) & 0xFF) - 127;
            ex = max(-126, min(126, 14 - e2));
          }
          const float sc = __uint_as_float((uint32_t)(ex + 127) << 23);
          const float inv = __uint_as_float((uint32_t)(127 - ex) << 23);
          for (int u = 0; u < D / 8; ++u) {
            const uint4 w = lds128(qrow + 16u * u);
            uint4 o;
            o.x = pack_f16(bf16_bits_to_f32(w.x & 0xFFFFu) * sc, bf16_bits_to_f32(w.x >> 16) * sc);
            o.y = pack_f16(bf16_bits_to_f32(w.y & 0xFFFFu) * sc, bf16_bits_to_f32(w.y >> 16) * sc);
            o.z = pack_f16(bf16_bits_to_f32(w.z & 0xFFFFu) * sc, bf16_bits_to_f32(w.z >> 16) * sc);
            o.w = pack_f16(bf16_bits_to_f32(w.w & 0xFFFFu) * sc, bf16_bits_to_f32(w.w >> 16) * sc);
            sts128(swz_unit(q16(), u / 8, kUmmaRows, rr, u % 8), o);
          }
          c = inv * p.sm_scale_log2 * (p.scale_mode == kScalePerTensor ? kscale : 1.f);
        } else {
          for (int u = 0; u < D / 8; ++u) sts128(swz_unit(q16(), u / 8, kUmmaRows, rr, u % 8), lds128(qrow + 16u * u));
          c = p.sm_scale_log2;
        }
      }
      row_c()[rr] = c;
      row_m()[rr] = rr < p.R ? -INFINITY : INFINITY;
      row_pos()[rr] = rr < p.R ? L - p.QL + rr / p.G : 0;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(sm.qempty(qs, p));
    o_valid = false;
    return true;
  }

  // One FP8 tensor of a stage -> FP16 operand ([chunks of 64 dims][TT rows]
  // [128 B], swizzled); V rows outside the stage's token range become zeros so
  // that poisoned slots never reach the MMA. Four units per pass, loads first.
  template <bool IS_V>
  __device__ void convert_tensor(uint32_t src_base, const StageView& h) {
    const uint32_t dst_base = sm.base_u32 + (IS_V ? p.off_v16 : p.off_k16);
    constexpr int UPR = NCH * 8;     // 16-byte FP8 units per token row
    constexpr int UNITS = TT * UPR;
    static_assert(UNITS % (4 * kUmmaThreads) == 0, "conversion passes");
#pragma unroll 1
    for (int e0 = threadIdx.x; e0 < UNITS; e0 += 4 * kUmmaThreads) {
      uint4 w[4];
      uint32_t dst[4];
      bool zero[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int ee = e0 + j * kUmmaThreads;
        const int t = ee / UPR, cb = (ee % UPR) / 8, c = ee % 8;
        w[j] = lds128(src_base + (uint32_t)(cb * TT + t) * 128u + (uint32_t)((c ^ (t & p.swz)) << 4));
        const int dim0 = cb * 128 + 16 * c;
        dst[j] = swz_unit(dst_base, dim0 / 64, TT, t, (dim0 % 64) / 8);
        zero[j] = IS_V && !(h.tbase + t >= h.t0 && h.tbase + t < h.t1);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint4 lo, hi;
        lo.x = e4m3x2_to_f16x2(w[j].x & 0xFFFFu);
        lo.y = e4m3x2_to_f16x2(w[j].x >> 16);
        lo.z = e4m3x2_to_f16x2(w[j].y & 0xFFFFu);
        lo.w = e4m3x2_to_f16x2(w[j].y >> 16);
        hi.x = e4m3x2_to_f16x2(w[j].z & 0xFFFFu);
        hi.y = e4m3x2_to_f16x2(w[j].z >> 16);
        hi.z = e4m3x2_to_f16x2(w[j].w & 0xFFFFu);
        hi.w = e4m3x2_to_f16x2(w[j].w >> 16);
        if (zero[j]) lo = hi = make_uint4(0, 0, 0, 0);
        // units u (even) and u + 1 of the same row: positions differ in bit 0
        sts128(dst[j], lo);
        sts128(dst[j] ^ 16u, hi);
      }
    }
  }

  // BF16 stage used in place: zero the V rows outside the token range.
  __device__ void clear_ragged_v(uint32_t vst, const StageView& h) {
    const int a = h.t0 - h.tbase, b = h.t1 - h.tbase;
    if (a <= 0 && b >= TT) return;
    for (int e = threadIdx.x; e < TT * NCH * 8; e += kUmmaThreads) {
      const int t = e / (NCH * 8);
      if (t >= a && t < b) continue;
      const int cb = (e % (NCH * 8)) / 8, c = e % 8;
      sts128(vst + (uint32_t)(cb * TT + t) * 128u + (uint32_t)(c << 4), make_uint4(0, 0, 0, 0));
    }
  }

  // Is (stage token t, row rr) visible? Rows past R are excluded by their
  // reference max (+inf), not here.
  __device__ __forceinline__ bool visible(const StageView& h, int t, int pos) const {
    const int tk = h.tbase + t;
    if (tk < h.t0 || tk >= h.t1) return false;
    if (p.causal && tk > pos) return false;
    if (p.window > 0 && tk <= pos - p.window) return false;
    return true;
  }

  // Load this thread's half of its token's S^T row (32 row scores).
  __device__ __forceinline__ void load_srow(float (&x)[kHalfRows]) {
    uint32_t v[32];
    tmem_ld32(tmem + lane_base + (uint32_t)(kHalfRows * half), v);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(v[i]);
    if constexpr (F8) {  // + the lo rows' partial scores
      tmem_ld32(tmem + lane_base + (uint32_t)(kUmmaRows + kHalfRows * half), v);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) x[i] += __uint_as_float(v[i]);
    }
  }

  // y[r] = score * c_r - m_r (log2 units, relative to the row's reference
  // max), -inf where masked; returns whether some visible y exceeds 8.
  __device__ __forceinline__ bool scaled_rows(const StageView& h, bool interior, float ks, float (&y)[kHalfRows]) {
    bool exceed = false;
    const bool tok_ok = tok >= 0;
    const int rb = kHalfRows * half;
#pragma unroll
    for (int r4 = 0; r4 < kHalfRows; r4 += 4) {
      const float4 c4 = *reinterpret_cast<const float4*>(row_c() + rb + r4);
      const float4 m4 = *reinterpret_cast<const float4*>(row_m() + rb + r4);
      const float cc[4] = {c4.x * ks, c4.y * ks, c4.z * ks, c4.w * ks};
      const float mm[4] = {m4.x, m4.y, m4.z, m4.w};
      int pos[4] = {0, 0, 0, 0};
      if (!interior) {
        const int4 p4 = *reinterpret_cast<const int4*>(row_pos() + rb + r4);
        pos[0] = p4.x;
        pos[1] = p4.y;
        pos[2] = p4.z;
        pos[3] = p4.w;
      }
      if (interior && tok_ok) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          y[r4 + i] = fmaf(y[r4 + i], cc[i], -mm[i]);
          exceed |= y[r4 + i] > 8.f;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float v = fmaf(y[r4 + i], cc[i], -mm[i]);
          const bool vis = tok_ok && (interior || visible(h, tok, pos[i]));
          y[r4 + i] = vis ? v : -INFINITY;
          exceed |= vis && v > 8.f;
        }
      }
    }
    return exceed;
  }

  // Slow path: raise the reference max of rows whose stage max exceeds it;
  // rescale O and L by 2^(m_old - m_new) in TMEM.
  __device__ void raise_max(const StageView& h, bool interior, float ks) {
    float x[kHalfRows];
    load_srow(x);
    const int rb = kHalfRows * half;
    // stage max of each row in absolute log2 units
#pragma unroll
    for (int r4 = 0; r4 < kHalfRows; r4 += 4) {
      const float4 c4 = *reinterpret_cast<const float4*>(row_c() + rb + r4);
      const float cc[4] = {c4.x * ks, c4.y * ks, c4.z * ks, c4.w * ks};
      int pos[4] = {0, 0, 0, 0};
      if (!interior) {
        const int4 p4 = *reinterpret_cast<const int4*>(row_pos() + rb + r4);
        pos[0] = p4.x;
        pos[1] = p4.y;
        pos[2] = p4.z;
        pos[3] = p4.w;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const bool vis = tok >= 0 && (interior || visible(h, tok, pos[i]));
        float v = vis ? x[r4 + i] * cc[i] : -INFINITY;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
        if (lane == 0) row_smax()[(warp & 3) * kUmmaRows + rb + r4 + i] = v;
      }
    }
    named_bar(1, kUmmaThreads);
    if (threadIdx.x < kUmmaRows) {
      const int rr = threadIdx.x;
      const float mold = row_m()[rr];
      float smax = row_smax()[rr];
#pragma unroll
      for (int w = 1; w < 4; ++w) smax = fmaxf(smax, row_smax()[w * kUmmaRows + rr]);
      float alpha = 1.f;
      if (smax > mold + 8.f) {  // false for rows past R (mold = +inf)
        if (mold != -INFINITY) alpha = ex2(mold - smax);
        row_m()[rr] = smax;
      }
      row_alpha()[rr] = alpha;
    }
    named_bar(1, kUmmaThreads);
    if (o_valid && half == 0) {
      // F8: every lane of the 128-row O holds a hi or lo part of row olane_row
      const float alpha = ((F8 || lane < 16) && olane_row < p.R) ? row_alpha()[olane_row] : 1.f;
      if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_base + kOCol + (uint32_t)c0, v);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
          tmem_st32(tmem + lane_base + kOCol + (uint32_t)c0, v);
        }
        uint32_t lv[32];  // L occupies the first 16 of these columns
        tmem_ld32(tmem + lane_base + kLCol, lv);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) lv[i] = __float_as_uint(__uint_as_float(lv[i]) * alpha);
        tmem_st32(tmem + lane_base + kLCol, lv);
        tmem_wait_st();
      }
    }
  }

  // Scores of this thread's token -> P^T row (16-bit, 128 bytes, swizzled).
  // every row's window is fully inside this stage's tokens?
  __device__ __forceinline__ bool interior_stage(const StageView& h) const {
    return flags()[1] != 0 && h.tbase >= h.t0 && h.tbase + TT <= h.t1 &&
           (!p.causal || h.tbase + TT - 1 <= flags()[2]) && (p.window == 0 || h.tbase > flags()[3] - p.window);
  }
  __device__ __forceinline__ float token_kscale(uint32_t sst) const {
    return (VTOK && tok >= 0) ? lds_f32(sst + 4u * tok) : 1.f;
  }

  // Scores -> P^T rows against the current reference max. Returns whether
  // some score exceeds its row's reference by more than 2^8 (the caller then
  // raises the max and calls this again).
  __device__ bool softmax_stage(const StageView& h, uint32_t sst) {
    const bool interior = interior_stage(h);
    const float ks = token_kscale(sst);
    float y[kHalfRows];
    load_srow(y);
    const bool exceed = scaled_rows(h, interior, ks, y);
    if (tok < 0) return exceed;
    // slots outside the token range may hold poisoned scales: P is 0 there
    const bool tok_in = h.tbase + tok >= h.t0 && h.tbase + tok < h.t1;
    const float vs = VTOK ? (tok_in ? lds_f32(sst + 4u * (TT + tok)) : 0.f) : 1.f;
    if constexpr (F8) {
      // P^T row of this token: bytes [0, 64) the rows' hi terms, [64, 128)
      // the lo terms; this thread's 32 rows are units 2h, 2h+1 and 4+2h, 5+2h
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        float e[16], hv[16], lv[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          e[i] = ex2(y[16 * g + i]);  // ex2(-inf) = +0
          const float pn = VTOK ? e[i] * vs : e[i];
          hv[i] = e4m3_lead(pn);
          lv[i] = pn - hv[i];
        }
        const int u = 2 * half + g;
        sts128(swz_unit(pt16(), 0, TT, tok, u),
               make_uint4(pack_e4m3x4(hv[0], hv[1], hv[2], hv[3]), pack_e4m3x4(hv[4], hv[5], hv[6], hv[7]),
                          pack_e4m3x4(hv[8], hv[9], hv[10], hv[11]), pack_e4m3x4(hv[12], hv[13], hv[14], hv[15])));
        sts128(swz_unit(pt16(), 0, TT, tok, 4 + u),
               make_uint4(pack_e4m3x4(lv[0], lv[1], lv[2], lv[3]), pack_e4m3x4(lv[4], lv[5], lv[6], lv[7]),
                          pack_e4m3x4(lv[8], lv[9], lv[10], lv[11]), pack_e4m3x4(lv[12], lv[13], lv[14], lv[15])));
        if constexpr (VTOK) {
          // the row sums take the plain P
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            hv[i] = e4m3_lead(e[i]);
            lv[i] = e[i] - hv[i];
          }
          sts128(swz_unit(pu16(), 0, TT, tok, u),
                 make_uint4(pack_e4m3x4(hv[0], hv[1], hv[2], hv[3]), pack_e4m3x4(hv[4], hv[5], hv[6], hv[7]),
                            pack_e4m3x4(hv[8], hv[9], hv[10], hv[11]), pack_e4m3x4(hv[12], hv[13], hv[14], hv[15])));
          sts128(swz_unit(pu16(), 0, TT, tok, 4 + u),
                 make_uint4(pack_e4m3x4(lv[0], lv[1], lv[2], lv[3]), pack_e4m3x4(lv[4], lv[5], lv[6], lv[7]),
                            pack_e4m3x4(lv[8], lv[9], lv[10], lv[11]), pack_e4m3x4(lv[12], lv[13], lv[14], lv[15])));
        }
      }
      return exceed;
    }
#pragma unroll
    for (int uu = 0; uu < 4; ++uu) {
      const int u = 4 * half + uu;  // 16-byte unit = rows 8u .. 8u + 7
      float e[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) e[i] = ex2(y[8 * uu + i]);  // ex2(-inf) = +0
      uint4 o, ou;
      if constexpr (FP8) {
        ou = make_uint4(pack_f16(e[0], e[1]), pack_f16(e[2], e[3]), pack_f16(e[4], e[5]), pack_f16(e[6], e[7]));
      } else {
        ou = make_uint4(pack_bf16(e[0], e[1]), pack_bf16(e[2], e[3]), pack_bf16(e[4], e[5]), pack_bf16(e[6], e[7]));
      }
      if constexpr (VTOK) {
        // the numerator takes P * v_scale(token); the row sums the plain P
        o = make_uint4(pack_f16(e[0] * vs, e[1] * vs), pack_f16(e[2] * vs, e[3] * vs), pack_f16(e[4] * vs, e[5] * vs),
                       pack_f16(e[6] * vs, e[7] * vs));
        sts128(swz_unit(pu16(), 0, TT, tok, u), ou);
      } else {
        o = ou;
      }
      sts128(swz_unit(pt16(), 0, TT, tok, u), o);
    }
    return exceed;
  }

  // Per-segment row facts used by the interior test: [1] all rows valid
  // (R == 64 is not needed: rows past R are excluded by their max), [2] the
  // smallest query position, [3] the largest.
  __device__ void segment_flags() {
    if (threadIdx.x == 0) {
      int lo = 1 << 30, hi = -(1 << 30);
      for (int rr = 0; rr < p.R; ++rr) {
        lo = min(lo, row_pos()[rr]);
        hi = max(hi, row_pos()[rr]);
      }
      flags()[1] = 1;
      flags()[2] = lo;
      flags()[3] = hi;
    }
  }

  // Descriptor of the operand byte_off bytes past a base descriptor's start
  // (the start field is the low 14 bits of address / 16; operands lie below
  // 256 KiB, so the add never carries out of it).
  __device__ __forceinline__ static uint64_t dadd(uint64_t d, uint32_t byte_off) { return d + (uint64_t)(byte_off >> 4); }

  __device__ void issue_s(uint64_t dk) {
    if constexpr (F8) {
      // K rows are 128 bytes = 128 e4m3 values: one chunk, 32-byte k-steps
#pragma unroll
      for (int j = 0; j < D / 32; ++j)
        umma_f8(tmem, dadd(dk, (uint32_t)j * 32u), dadd(dq, (uint32_t)j * 32u), kIdescS, j > 0 ? 1u : 0u);
    } else {
#pragma unroll
      for (int j = 0; j < D / 16; ++j) {
        const uint64_t ad = dadd(dk, (uint32_t)(j / 4) * (TT * 128u) + (uint32_t)(j % 4) * 32u);
        const uint64_t bd = dadd(dq, (uint32_t)(j / 4) * (kUmmaRows * 128u) + (uint32_t)(j % 4) * 32u);
        umma_f16(tmem, ad, bd, kIdescS, j > 0 ? 1u : 0u);
      }
    }
    umma_commit(sbar_addr);
  }
  __device__ void issue_pv(uint64_t dv, bool accumulate) {
    if constexpr (F8) {
      // A = P^T [TT tokens][128 hi/lo rows], B = V [TT tokens][128 dims]:
      // both MN-major e4m3, 32 tokens (4 KiB) per k-step
#pragma unroll
      for (int j = 0; j < TT / 32; ++j)
        umma_f8(tmem + kOCol, dadd(dpt, (uint32_t)j * 4096u), dadd(dv, (uint32_t)j * 4096u), kIdescPV,
                (accumulate || j > 0) ? 1u : 0u);
#pragma unroll
      for (int j = 0; j < TT / 32; ++j)
        umma_f8(tmem + kLCol, dadd(VTOK ? dpu : dpt, (uint32_t)j * 4096u), dadd(dones, (uint32_t)j * 32u), kIdescL,
                (accumulate || j > 0) ? 1u : 0u);
      umma_commit(obar_addr);
      return;
    }
    // A = P^T stored [TT tokens][64 rows]: MN-major, one 64-row chunk;
    // B = V [TT tokens][D]: MN-major, D/64 chunks of TT*128 bytes
#pragma unroll
    for (int j = 0; j < TT / 16; ++j)
      umma_f16(tmem + kOCol, dadd(dpt, (uint32_t)j * 2048u), dadd(dv, (uint32_t)j * 2048u), kIdescPV,
               (accumulate || j > 0) ? 1u : 0u);
#pragma unroll
    for (int j = 0; j < TT / 16; ++j)
      umma_f16(tmem + kLCol, dadd(VTOK ? dpu : dpt, (uint32_t)j * 2048u),
               dadd(dones, (uint32_t)(j / 4) * (16 * 128u) + (uint32_t)(j % 4) * 32u), kIdescL,
               (accumulate || j > 0) ? 1u : 0u);
    umma_commit(obar_addr);
  }

  __device__ void end_segment(const StageView& h, int slot, const MergeDesc& md) {
    if (pv_pending) wait_pv();
    const bool whole = (h.flags & kSegWhole) != 0;
    const bool cluster = p.merge == kMergeCluster;
    float* cp_o = reinterpret_cast<float*>(sm.base + p.off_cpart);
    float* cp_ml = cp_o + (size_t)p.Rpad * D;
    const float M = row_own ? row_m()[r] : -INFINITY;
    // write 32 columns of this thread's row (row_own threads)
    auto emit = [&](int c0, const float* v, float L) {
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        const float4 f = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
        const int d = c0 + i;
        if (whole)
          finalize_store<D>(p, vscale, f, M, L, h.b, h.g, r, d);
        else if (cluster)
          *reinterpret_cast<float4*>(cp_o + (size_t)r * D + d) = f;
        else
          *reinterpret_cast<float4*>(p.part_o + ((size_t)slot * p.Rpad + r) * D + d) = f;
      }
    };
    float L = 0.f;
    if constexpr (F8) {
      // O and L rows are hi part (lanes 0..63) + lo part (lanes 64..127):
      // quarters 2, 3 pass theirs through shared memory (the P^T buffer, idle
      // now) 32 columns at a time
      float* scr = reinterpret_cast<float*>(sm.base + p.off_p16);  // [64 rows][33]
      const bool lo_part = half == 0 && (warp & 3) >= 2;
      const bool hi_part = half == 0 && (warp & 3) < 2;
      uint32_t lv[32];
      if (o_valid && half == 0) {
        tmem_ld32(tmem + lane_base + kLCol, lv);
        tmem_wait_ld();
      }
      if (lo_part) scr[64 * 33 + olane_row] = o_valid ? __uint_as_float(lv[0]) : 0.f;
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t v[32];
        if (o_valid && half == 0) {
          tmem_ld32(tmem + lane_base + kOCol + (uint32_t)c0, v);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0u;
        }
        if (lo_part) {
#pragma unroll
          for (int i = 0; i < 32; ++i) scr[olane_row * 33 + i] = __uint_as_float(v[i]);
        }
        named_bar(1, kUmmaThreads);
        if (hi_part) {
          if (c0 == 0) L = (o_valid ? __uint_as_float(lv[0]) : 0.f) + scr[64 * 33 + olane_row];
          float f[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(v[i]) + scr[olane_row * 33 + i];
          if (row_own) emit(c0, f, L);
        }
        named_bar(1, kUmmaThreads);
      }
    } else {
      if (o_valid && half == 0) {
        uint32_t lv[32];
        tmem_ld32(tmem + lane_base + kLCol, lv);
        tmem_wait_ld();
        L = __uint_as_float(lv[0]);
      }
#pragma unroll 1
      for (int c0 = 0; c0 < D && half == 0; c0 += 32) {
        uint32_t v[32];
        if (o_valid) {
          tmem_ld32(tmem + lane_base + kOCol + (uint32_t)c0, v);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0u;
        }
        if (!row_own) continue;
        float f[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(v[i]);
        emit(c0, f, L);
      }
    }
    if (row_own && !whole) {
      const float2 ml = make_float2(M, L);
      if (cluster)
        *reinterpret_cast<float2*>(cp_ml + 2 * r) = ml;
      else
        *reinterpret_cast<float2*>(p.part_ml + ((size_t)slot * p.Rpad + r) * 2) = ml;
    }
    // O and L are read; the next segment's first PV may overwrite them
    tc_fence_before();
    if (whole || cluster) return;
    if (p.merge == kMergeReducer) {
      if (threadIdx.x == 0 && slot == md.s0) p.unit_desc[h.unit] = make_int4(md.nseg, md.s0, md.sbase, md.sstride);
    } else if (p.merge == kMergeLastArriver) {
      __threadfence();
      named_bar(1, kUmmaThreads);
      if (threadIdx.x == 0) la_arrive(p, sm, h.b, h.g, h.unit, md);
      named_bar(1, kUmmaThreads);
      la_run_queue<D>(p, sm, vscale, kUmmaThreads);
    }
  }

  __device__ void run() {
    setup();
    int n = 0;
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
      if (h.flags & kSegFirst) {
        if (!begin_segment(h.L)) {
          fail();
          break;
        }
        named_bar(1, kUmmaThreads);  // row state written
        segment_flags();
      }
      const uint32_t kst = sm.stage(s, p);
      const uint32_t vst = kst + (uint32_t)TT * 128u * NCH;
      const uint32_t sst = kst + p.off_scale;
      const bool has_tokens = h.t1 > h.t0;
      if (!has_tokens) {
        __syncwarp();
        if (lane == 0) mbar_arrive(sm.empty(s, p));
      } else {
        // K operand (the previous S chain, its only reader, has completed);
        // the previous PV may still run meanwhile
        if constexpr (CONV) convert_tensor<false>(kst, h);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        tc_fence_before();
        named_bar(1, kUmmaThreads);
        if (threadIdx.x == 0) {
          tc_fence_after();
          issue_s(CONV ? dk16 : umma_sdesc(kst, 16, 1024));
        }
        // V and P are rewritten only after the previous PV has completed; the
        // V conversion overlaps the S chain
        if (pv_pending) wait_pv();
        if constexpr (CONV)
          convert_tensor<true>(vst, h);
        else
          clear_ragged_v(vst, h);
        if (CONV && !VTOK) {
          // this warp is done with the stage's bytes
          __syncwarp();
          if (lane == 0) mbar_arrive(sm.empty(s, p));
        }
        if (!mbar_wait_spin(sbar(), ph_s)) fail();
        ph_s ^= 1u;
        tc_fence_after();
        bool exceed = softmax_stage(h, sst);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        tc_fence_before();
        if (named_bar_or(1, kUmmaThreads, exceed)) {
          // rare: a row's max moved past its reference; raise it (rescaling
          // O and L) and recompute this stage's P
          raise_max(h, interior_stage(h), token_kscale(sst));
          (void)softmax_stage(h, sst);
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          tc_fence_before();
          named_bar(1, kUmmaThreads);
        }
        if (CONV && VTOK) {
          __syncwarp();
          if (lane == 0) mbar_arrive(sm.empty(s, p));
        }
        if (threadIdx.x == 0) {
          tc_fence_after();
          issue_pv(CONV ? dv16 : umma_sdesc(vst, TT * 128u, 1024), o_valid);
        }
        pv_pending = true;
        o_valid = true;
        if (!CONV) pend_stage = s;  // the MMAs read this stage in place
      }
      if (h.flags & kSegLast) end_segment(h, slot, md);
      ++n;
    }
    teardown();
  }
};

// Producer warp = warp 8; consumer warps 0..7.
template <bool FP8, int D, bool VTOK>
__global__ void __launch_bounds__(288, 1) pa_umma_kernel(const __grid_constant__ PaParams p,
                                                         const __grid_constant__ CUtensorMap tmK,
                                                         const __grid_constant__ CUtensorMap tmV) {
  extern __shared__ uint8_t smem_raw[];
  Smem sm;
  {
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t aligned = (raw + 1023u) & ~1023u;
    sm.base = smem_raw + (aligned - raw);
    sm.base_u32 = aligned;
  }
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.NS; ++s) {
      mbar_init(sm.full(s, p), 1);
      mbar_init(sm.empty(s, p), p.NCW);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(sm.qfull(i, p), 1);
      mbar_init(sm.qempty(i, p), p.NCW);
    }
    mbar_init(sm.base_u32 + p.off_ubar, 1);
    mbar_init(sm.base_u32 + p.off_ubar + 8, 1);
    for (int i = 0; i < 16; ++i) sm.misc(p)[i] = 0;
    fence_barrier_init();
  }
  __syncthreads();
  constexpr int ELT = FP8 ? 1 : 2;
  constexpr int NCH = D * ELT / 128;
  if (warp == p.NCW) {
    Producer<ELT, NCH> prod(p, &tmK, &tmV, sm);
    prod.run();
    if (p.merge == kMergeCluster) {
      cluster_sync_all();
      cluster_sync_all();
    }
  } else {
    UmmaConsumer<FP8, D, VTOK> cons(p, sm);
    cons.run();
    if (p.merge == kMergeCluster) {
      cluster_sync_all();
      cluster_merge_unit<D>(p, sm, cons.vscale, blockIdx.x / p.P, threadIdx.x, kUmmaThreads);
      cluster_sync_all();
    }
  }
}

}  // namespace dev
}  // namespace pa
