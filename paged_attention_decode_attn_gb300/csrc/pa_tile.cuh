// Split-KV paged-attention decode tile kernel for sm_103a.
//
// Roles inside one CTA:
//  * one producer warp walks the CTA's share of (sequence, KV head) token
//    chunks, stages block-table page ids in its registers (32 per coalesced
//    load, the next batch prefetched), and fills a ring of shared-memory
//    stages with TMA copies (cp.async.bulk.tensor, 128-byte swizzle; sparse
//    rows with 16-byte cp.async in the same swizzle), completing on mbarriers;
//  * NCW consumer warps read each stage, compute S^T = K Q^T and O^T += V^T P^T
//    with mma.sync m16n8k16 (tokens or head dims on the M side, query rows on
//    the N side, so a GQA8 group fills the 8-wide N tile exactly), scale and
//    mask the scores, keep the online softmax in registers (warp shuffles), and
//    at each segment end merge their token groups and either write the BF16
//    output or a partial (max, sum, unnormalised O) that the last-arriver,
//    cluster or reducer merge combines in partition order.
//
// Sources of the method: PR "Add paged-attention Tile kernel" (API, layouts,
// per-tensor/per-token scales, split partitions and their reduction), PR
// "Extend packed D256 PA decode pipe to page16, transposed V and sliding
// windows" (page-id staging, window-bounded page ranges, scale before mask,
// per-token scales, MTP rows), PR "Merge gfx1250 PA decode partitions in the
// tile kernel and speed up dense decode" (cluster merge, last-arriver merge
// with self-resetting arrival counters, row scale folded into the exponent,
// interior tiles without masks, double-buffered pages with asynchronous scale
// copies).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "pa_internal.h"

namespace pa {
namespace dev {

constexpr float kLog2e = 1.4426950408889634f;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s per wait

// Stage header written by the producer before it arms the stage. Consumers
// read the first 32 bytes on every stage (48 for sparse), the rest only at
// segment boundaries.
struct alignas(16) StageHdr {
  int kind_flags;  // kSeg* flags; kEnd marks the end of the CTA's work
  int tbase;       // token (sparse: index position) of stage row 0
  int t0, t1;      // rows [t0 - tbase, t1 - tbase) carry real tokens of the visible range
  int L;           // context length of the sequence
  int unit, b, g;  // (sequence, KV head) unit
  unsigned mask[4];  // sparse: validity of stage rows 0..127
  int slot;          // partial slot of this segment
  int nseg, s0, sbase;
  int sstride;       // merge slot list: k == 0 -> s0, else sbase + k * sstride
  int pad[15];
};
static_assert(sizeof(StageHdr) == 128, "header size");
constexpr int kEnd = 1 << 8;
constexpr int kScanRegs = 8;       // schedule scan in registers for batch <= 256
constexpr int kMaxTokenWarps = 4;  // token groups per CTA (the plan never makes more)

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, int count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint32_t bar, uint32_t tx) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(tx)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  // The suspend-time hint lets the warp sleep until the phase completes
  // instead of spinning on the barrier.
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(1000000u)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ unsigned long long global_timer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Bounded wait on a phase; false after ~2 s (the caller records a timeout).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 4; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_timer() - t0 > kWaitLimitNs) return false;
  }
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* tm, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
// 16-byte (L2-only) and 4-byte asynchronous copies to shared memory; the
// noinc arrive fires on `bar` once every copy this thread issued so far has
// landed, without raising the barrier's expected count (it is part of it).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* tm) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tm)) : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ int4 lds128i(uint32_t addr) {
  int4 v;
  asm volatile("ld.shared.v4.s32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ float lds_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ void named_bar(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
  uint32_t r;
  uint16_t v = static_cast<uint16_t>(two_bytes & 0xFFFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
  return r;
}
// Two OCP FP4 E2M1 codes (the low byte of x, first element in the low
// nibble) as FP16x2, first element in the low half; every E2M1 value is exact
// in FP16.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t x) {
  uint32_t r;
  asm("{\n .reg .b8 b;\n mov.b32 {b, _, _, _}, %1;\n cvt.rn.f16x2.e2m1x2 %0, b;\n}\n" : "=r"(r) : "r"(x));
  return r;
}
__device__ __forceinline__ uint32_t mul_f16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
// MX block scales of one head_dim-128 token row: four E8M0 bytes (blocks of
// 32 dims, first block in the low byte). The row is taken in units of its
// largest scale: 2^(max - 127) as binary32 (NaN for the NaN code 0xFF) ...
__device__ __forceinline__ int mx_max_code(uint32_t w) {
  return max(max((int)(w & 0xFFu), (int)((w >> 8) & 0xFFu)), max((int)((w >> 16) & 0xFFu), (int)(w >> 24)));
}
__device__ __forceinline__ float e8m0_to_f32(int x) {
  if (x == 0xFF) return __uint_as_float(0x7FC00000u);
  return x == 0 ? __uint_as_float(0x00400000u) : __uint_as_float((uint32_t)x << 23);
}
// ... and each block's elements are multiplied in FP16 by 2^(code - max) =
// 2^-d: exact down to 2^-24 (FP16 subnormals), 0 for d > 24 (a block more than
// 2^24 below the row's largest).
__device__ __forceinline__ uint32_t f16x2_pow2_neg(int d) {
  uint32_t h = d <= 14 ? (uint32_t)(15 - d) << 10 : (d <= 24 ? 1u << (24 - d) : 0u);
  return h | (h << 16);
}
__device__ __forceinline__ uint32_t mx_block_factor(uint32_t w, int blk) {
  return f16x2_pow2_neg(mx_max_code(w) - (int)((w >> (8 * blk)) & 0xFFu));
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t movm_trans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}
template <bool F16>
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  if constexpr (F16) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t bits16) { return __uint_as_float(bits16 << 16); }
__device__ __forceinline__ float f16_bits_to_f32(uint32_t bits16) {
  return __half2float(__ushort_as_half((unsigned short)bits16));
}
// A query element (BF16 or FP16 bits in the low half of the word), widened exactly.
__device__ __forceinline__ float q_bits_to_f32(uint32_t bits16, bool f16) {
  return f16 ? f16_bits_to_f32(bits16) : bf16_bits_to_f32(bits16);
}
// Two output elements in the queries' type (round to nearest even).
__device__ __forceinline__ uint32_t pack_out(float lo, float hi, bool f16) {
  return f16 ? pack_f16(lo, hi) : pack_bf16(lo, hi);
}

// ------------------------------------------------------- schedule arithmetic
// Visible token range of sequence b as a chunk range (union over the QL rows).
struct UnitRange {
  int L, lo, hi, c_lo, n;  // n = chunks touching [lo, hi) (0 if empty)
};
__device__ __forceinline__ UnitRange unit_range(const PaParams& p, int b) {
  UnitRange r;
  int L = __ldg(p.ctx_lens + b);
  L = max(0, min(L, p.maxp * p.S));
  r.L = L;
  if (p.topk > 0) {
    r.lo = 0;
    r.hi = p.topk;
    r.c_lo = 0;
    r.n = (p.topk + p.TT - 1) / p.TT;
    return r;
  }
  int lo = 0;
  if (p.window > 0) lo = max(0, L - p.QL + 1 - p.window);
  r.lo = lo;
  r.hi = L;
  if (L > lo) {
    r.c_lo = lo / p.TT;
    r.n = (L + p.TT - 1) / p.TT - r.c_lo;
  } else {
    r.c_lo = 0;
    r.n = 0;
  }
  return r;
}
// Balanced schedule: chunk x of the global list belongs to CTA owner(x);
// CTA c starts at start(c) = floor(c * N / C).
__device__ __forceinline__ long long sched_start(long long c, long long N, long long C) { return c * N / C; }
__device__ __forceinline__ long long sched_owner(long long x, long long N, long long C) {
  return ((x + 1) * C - 1) / N;
}
// Weight of sequence b in the balanced schedule: each of its units counts its
// chunks (at least one) plus seg_cost virtual chunks that stand for the fixed
// cost of a segment. The virtual chunks come first in the unit's range and
// carry no work, so a CTA whose range holds many short units gets fewer real
// chunks.
__device__ __forceinline__ long long seq_weight(const PaParams& p, int b) {
  return (long long)p.Hkv * (max(1, unit_range(p, b).n) + p.seg_cost);
}
// Total weight of the balanced schedule (warp-collective).
__device__ __forceinline__ long long balanced_total(const PaParams& p, int lane) {
  long long tot = 0;
  // unrolled so that several rounds' length loads are in flight together
#pragma unroll 8
  for (int b0 = 0; b0 < p.B; b0 += 32) {
    int b = b0 + lane;
    long long cnt = 0;
    if (b < p.B) cnt = seq_weight(p, b);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, off);
    tot += cnt;
  }
  return tot;
}
// Sequence containing global chunk x and the chunk count before it (warp-collective).
__device__ __forceinline__ void balanced_find(const PaParams& p, int lane, long long x, int& b_out, long long& excl_out) {
  long long base = 0;
  b_out = p.B;
  excl_out = base;
  for (int b0 = 0; b0 < p.B; b0 += 32) {
    int b = b0 + lane;
    long long cnt = 0;
    if (b < p.B) cnt = seq_weight(p, b);
    long long incl = cnt;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      long long v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    long long total = __shfl_sync(0xffffffffu, incl, 31);
    unsigned hit = __ballot_sync(0xffffffffu, b < p.B && base + incl > x);
    if (hit) {
      int first = __ffs(hit) - 1;
      long long ex = __shfl_sync(0xffffffffu, incl - cnt, first);
      b_out = b0 + first;
      excl_out = base + ex;
      return;
    }
    base += total;
  }
}
// Merge descriptor of a unit whose weight range starts at Pu and whose nu real
// chunks start at Pu + A. CTAs c1..c2 own the real chunks; c1 writes slot
// 2*c1 + 1 if its range began before Pu (it then holds the previous unit's
// last chunk), else 2*c1; the others write 2*c.
struct MergeDesc {
  int nseg, s0, sbase, sstride;
};
__device__ __forceinline__ MergeDesc balanced_desc(long long Pu, long long nu, long long A, long long N, long long C) {
  MergeDesc d;
  long long c1 = sched_owner(Pu + A, N, C), c2 = sched_owner(Pu + A + nu - 1, N, C);
  d.nseg = (int)(c2 - c1 + 1);
  d.s0 = (int)(2 * c1 + (sched_start(c1, N, C) < Pu ? 1 : 0));
  d.sbase = (int)(2 * c1);
  d.sstride = 2;
  return d;
}
__device__ __forceinline__ int merge_slot(const MergeDesc& d, int k) { return k == 0 ? d.s0 : d.sbase + k * d.sstride; }

// ------------------------------------------------------------ shared layout
struct Smem {
  uint8_t* base;
  uint32_t base_u32;
  __device__ __forceinline__ uint32_t stage(int s, const PaParams& p) const {
    return base_u32 + p.off_stage + s * p.stage_bytes;
  }
  __device__ __forceinline__ StageHdr* hdr(int s, const PaParams& p) const {
    return reinterpret_cast<StageHdr*>(base + p.off_hdr) + s;
  }
  __device__ __forceinline__ uint32_t hdr_u32(int s, const PaParams& p) const {
    return base_u32 + p.off_hdr + 128u * s;
  }
  __device__ __forceinline__ uint32_t full(int s, const PaParams& p) const { return base_u32 + p.off_bar + 8 * s; }
  __device__ __forceinline__ uint32_t empty(int s, const PaParams& p) const {
    return base_u32 + p.off_bar + 8 * (p.NS + s);
  }
  // Q ring: slot i's rows arrive on qfull(i); qempty(i) collects one arrival
  // per consumer warp once the rows are in registers.
  __device__ __forceinline__ uint32_t qfull(int i, const PaParams& p) const {
    return base_u32 + p.off_bar + 16 * p.NS + 8 * i;
  }
  __device__ __forceinline__ uint32_t qempty(int i, const PaParams& p) const {
    return base_u32 + p.off_bar + 16 * p.NS + 16 + 8 * i;
  }
  __device__ __forceinline__ uint32_t qbuf(int i, const PaParams& p) const {
    return base_u32 + p.off_q + i * p.q_slot_bytes;
  }
  __device__ __forceinline__ volatile int* misc(const PaParams& p) const {
    return reinterpret_cast<volatile int*>(base + p.off_misc);
  }
};

// Read one field from each 64-byte line of the kernel parameters, all before
// any is used: the first access to a line misses the constant cache and,
// after L2 has been evicted, goes to DRAM; issued together the misses overlap
// instead of stalling the producer's control flow one line at a time.
__device__ __forceinline__ void prefetch_params(const PaParams& p) {
  static_assert(sizeof(PaParams) <= 6 * 64, "one field per parameter line below");
  const uint64_t a0 = reinterpret_cast<uint64_t>(p.out);
  const uint64_t a1 = reinterpret_cast<uint64_t>(p.part_o);
  const int a2 = p.B, a3 = p.window, a4 = p.C, a5 = p.off_hdr, a6 = p.off_q, a7 = p.off_rows;
  asm volatile("" ::"l"(a0), "l"(a1), "r"(a2), "r"(a3), "r"(a4), "r"(a5), "r"(a6), "r"(a7));
}

__device__ __forceinline__ void flag_status(const PaParams& p, int bits) {
  if (p.status) atomicOr(p.status, bits);
}

// ------------------------------------------------------------ merge math
// out = O * (1/L) (* per-tensor V scale), with an optional sink logit added to
// the denominator (natural-log units, converted to log2 here).
template <int D>
__device__ __forceinline__ void finalize_store(const PaParams& p, float vscale, float4 O, float M, float L, int b,
                                               int g, int r, int d) {
  const int i = r / p.G;
  const int head = g * p.G + r % p.G;
  if (p.has_sinks) {
    const float s2 = __ldg(p.sinks + head) * kLog2e;
    const float M2 = fmaxf(M, s2);
    const float a = (M == -INFINITY) ? 0.f : ex2(M - M2);
    L = fmaf(L, a, ex2(s2 - M2));
    O.x *= a;
    O.y *= a;
    O.z *= a;
    O.w *= a;
  }
  const float inv = (L > 0.f) ? (1.f / L) * vscale : 0.f;
  uint2 st;
  st.x = pack_out(O.x * inv, O.y * inv, p.q_f16 != 0);
  st.y = pack_out(O.z * inv, O.w * inv, p.q_f16 != 0);
  *reinterpret_cast<uint2*>(p.out + ((size_t)(b * p.QL + i) * p.Hq + head) * D + d) = st;
}

// Merge n partials (max, sum, O) in order q = 0..n-1 for output elements
// [e0, e1) (groups of 4 head dims, row-major over the unit's rows) and store
// the BF16 rows. Every merge path (last arriver, cluster, reducer) goes
// through this function with the same partial order, so they agree bit for bit.
template <int D, class LoadML, class LoadO>
__device__ __forceinline__ void merge_elems(const PaParams& p, float vscale, int n, int b, int g, int tid, int nthr,
                                            int e0, int e1, LoadML load_ml, LoadO load_o) {
  // Partials are read in chunks of kChunk whose loads are all issued before
  // any is used (one memory round trip per chunk); chunks fold into a running
  // (max, sum, O) in partition order. An empty partial (max = -inf, sum = 0,
  // O = 0) contributes exact zeros.
  constexpr int kChunk = 8;
  for (int e = e0 + tid; e < e1; e += nthr) {
    const int r = e / (D / 4);
    const int d = (e % (D / 4)) * 4;
    float M = -INFINITY, L = 0.f;
    float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int q0 = 0; q0 < n; q0 += kChunk) {
      float2 ml[kChunk];
      float4 ov[kChunk];
#pragma unroll
      for (int q = 0; q < kChunk; ++q) {
        if (q0 + q < n) {
          ml[q] = load_ml(q0 + q, r);
          ov[q] = load_o(q0 + q, r, d);
        } else {
          ml[q] = make_float2(-INFINITY, 0.f);
          ov[q] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      float Mc = M;
#pragma unroll
      for (int q = 0; q < kChunk; ++q) Mc = fmaxf(Mc, ml[q].x);
      if (Mc == -INFINITY) continue;
      const float c = ex2(M - Mc);  // rescale what the earlier chunks summed (0 if none)
      L *= c;
      O.x *= c;
      O.y *= c;
      O.z *= c;
      O.w *= c;
#pragma unroll
      for (int q = 0; q < kChunk; ++q) {
        const float a = ex2(ml[q].x - Mc);
        L = fmaf(ml[q].y, a, L);
        O.x = fmaf(ov[q].x, a, O.x);
        O.y = fmaf(ov[q].y, a, O.y);
        O.z = fmaf(ov[q].z, a, O.z);
        O.w = fmaf(ov[q].w, a, O.w);
      }
      M = Mc;
    }
    finalize_store<D>(p, vscale, O, M, L, b, g, r, d);
  }
}


__device__ __forceinline__ float per_tensor_vscale(const PaParams& p) {
  return p.scale_mode == kScalePerTensor ? __ldg(p.v_scale) : 1.f;
}

// ================================================================ producer
// ROWB: bytes of one stage row per column block (128; 64 for MXFP4 head_dim
// 128, whose rows the 64-byte swizzle lays out).
template <int ELT, int NCH, int ROWB = 128>
struct Producer {
  const PaParams& p;
  const CUtensorMap* tmK;
  const CUtensorMap* tmV;
  Smem sm;
  int lane;
  int n = 0;  // stages filled so far
  bool ok = true;
  // page-id staging: lane l holds the physical page of logical page pbase + l
  int pid_b = -1, pbase = 0, pid_cur = -1, pid_next = -1, npages_b = 0;
  // the window a unit's walk began at, kept for the next KV head of the same
  // sequence (same block-table row, same start)
  int first_base = 0, first_cur = -1, first_next = -1;

  __device__ __forceinline__ Producer(const PaParams& p_, const CUtensorMap* k, const CUtensorMap* v, Smem s)
      : p(p_), tmK(k), tmV(v), sm(s), lane(threadIdx.x & 31) {}

  __device__ __forceinline__ int load_pid(int b, int lp) const {
    if (lp < 0 || lp >= npages_b) return -1;
    return __ldg(p.block_table + (size_t)b * p.maxp + lp);
  }
  // Make the batch of 32 page ids holding logical page lp0 current (loads
  // are issued here and waited for at first use).
  __device__ __forceinline__ void stage_window(int b, int L, int lp0, int align) {
    if (b != pid_b) {
      pid_b = b;
      npages_b = (L + p.S - 1) / p.S;
      pbase = -(1 << 30);
      first_base = -(1 << 30);
    }
    if (lp0 < pbase || lp0 >= pbase + 32) {
      if (lp0 >= pbase + 32 && lp0 < pbase + 64) {
        pid_cur = pid_next;
        pbase += 32;
        pid_next = load_pid(b, pbase + 32 + lane);
      } else if (lp0 - lp0 % align == first_base) {
        pbase = first_base;
        pid_cur = first_cur;
        pid_next = first_next;
      } else {
        pbase = lp0 - lp0 % align;
        pid_cur = load_pid(b, pbase + lane);
        pid_next = load_pid(b, pbase + 32 + lane);
        first_base = pbase;
        first_cur = pid_cur;
        first_next = pid_next;
      }
    }
  }
  // Physical page of logical page lp0 + lane (lanes < pages in the stage; the
  // stage's pages lie inside one aligned batch of 32).
  __device__ __forceinline__ int staged_pages(int b, int L, int lp0, int align) {
    stage_window(b, L, lp0, align);
    return __shfl_sync(0xffffffffu, pid_cur, (lp0 - pbase + lane) & 31);
  }

  __device__ __forceinline__ bool acquire_stage(int& s) {
    s = n % p.NS;
    const uint32_t par = ((n / p.NS) & 1) ^ 1;
    bool got = mbar_wait(sm.empty(s, p), par);
    got = __all_sync(0xffffffffu, got);
    if (!got) {
      ok = false;
      if (lane == 0) {
        flag_status(p, kStatusTimeout);
        sm.misc(p)[0] = 1;
      }
    }
    return got;
  }

  __device__ __forceinline__ void emit_dense(const StageHdr& h) {
    int s;
    if (!acquire_stage(s)) return;
    const int S = p.S, TT = p.TT, BH = p.BH;
    int nbox = 0, lp0 = 0, row0 = 0, yoff = 0;
    if (h.t1 > h.t0) {
      if (S >= TT) {
        nbox = 1;
        lp0 = h.tbase / S;
        yoff = h.tbase % S;
        row0 = 0;
      } else {
        lp0 = h.t0 / S;
        nbox = (h.t1 - 1) / S - lp0 + 1;
        row0 = lp0 * S - h.tbase;
      }
    }
    int phys = 0;
    if (nbox > 0) phys = staged_pages(h.b, h.L, lp0, S < TT ? TT / S : 1);
    const bool ktok = p.scale_mode == kScalePerToken;
    const uint32_t bytes = (uint32_t)nbox * BH * (uint32_t)ROWB * NCH * 2u + (ktok ? (uint32_t)nbox * BH * 8u : 0u);
    if (lane == 0) {
      *sm.hdr(s, p) = h;
      if (bytes)
        mbar_arrive_tx(sm.full(s, p), bytes);
      else
        mbar_arrive(sm.full(s, p));
    }
    __syncwarp();
    if (lane < nbox) {
      if (phys < 0 || phys >= p.num_pages) {
        flag_status(p, kStatusBadPage);
        phys = 0;
      }
      const int y = (phys * p.Hkv + h.g) * S + yoff;
      const int row = row0 + lane * BH;
      const uint32_t kst = sm.stage(s, p);
      const uint32_t vst = kst + (uint32_t)TT * (uint32_t)ROWB * NCH;
      const uint32_t bar = sm.full(s, p);
#pragma unroll
      for (int cb = 0; cb < NCH; ++cb)
        tma_load_2d(kst + (uint32_t)(cb * TT + row) * (uint32_t)ROWB, tmK, cb * (128 / ELT), y, bar);
      if (p.v_tr) {
        // transposed V: the page's chunks of 8 tokens ([D][8] BF16 each) as
        // 128-byte rows of 8 dims; the stage holds chunk after chunk
        tma_load_2d(vst + (uint32_t)row * (uint32_t)(2 * p.D), tmV, 0, y * (p.D / 64), bar);
      } else {
#pragma unroll
        for (int cb = 0; cb < NCH; ++cb)
          tma_load_2d(vst + (uint32_t)(cb * TT + row) * (uint32_t)ROWB, tmV, cb * (128 / ELT), y, bar);
      }
      if (ktok) {
        const uint32_t sc = kst + p.off_scale;
        bulk_load(sc + row * 4, p.k_scale + y, BH * 4, bar);
        bulk_load(sc + TT * 4 + row * 4, p.v_scale + y, BH * 4, bar);
      }
    }
  }

  // Sparse stages: row r of stage k holds index position tbase + r. Loads
  // run ahead of the stages: when stage k's gathers are issued, the page ids
  // of stage k+1 (whose indices arrived meanwhile) and the indices of stage
  // k+2 are requested, so a stage rarely waits on a block-table round trip.
  int la_b = -1, la_pos = -1;  // stage whose indices and page ids are requested
  int la_idx[4], la_phys[4];
  int nx_b = -1, nx_pos = -1;  // stage whose indices are requested
  int nx_idx[4];

  __device__ __forceinline__ void load_phys(int b, int L, const int* idx, int* phys) const {
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const int t = idx[rr];
      phys[rr] = (t >= 0 && t < L) ? __ldg(p.block_table + (size_t)b * p.maxp + t / p.S) : -1;
    }
  }
  // Request the indices of the stage at index position pos of sequence b.
  __device__ __forceinline__ void request_indices(int b, int pos) {
    nx_b = b;
    nx_pos = pos;
    load_indices(b, pos, p.topk, nx_idx);
  }

  __device__ __forceinline__ void load_indices(int b, int pos0, int pos_end, int* idx) const {
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const int row = rr * 32 + lane;
      const int pos = pos0 + row;
      idx[rr] = (row < p.TT && pos < pos_end) ? __ldg(p.topk_idx + (size_t)b * p.topk + pos) : -1;
    }
  }

  // Copy the valid rows of a sparse stage into its K and V buffers with
  // 16-byte asynchronous copies. Stage row r (r < TTC = 128 / NCH tokens)
  // owns chunk rows cb * TTC + r, one per 128-byte column block cb; each
  // instruction moves four whole chunk rows (eight lanes per row), written
  // in the 128-byte swizzle the consumers read (16-byte piece j of chunk
  // row c at piece j ^ (c & 7)). Lane l holds the cache row y and the
  // validity of stage rows l, 32 + l, ... (yv, mask). Rows without a token
  // are not copied: their scores are masked and their V rows zeroed.
  __device__ __forceinline__ void gather_rows(uint32_t kst, uint32_t vst, const int (&yv)[4], const unsigned (&mask)[4]) {
    constexpr int TTC = 128 / NCH;
    constexpr int kRowBytes = 128 * NCH;
    const int j = lane & 7, rq = lane >> 3;
    const uint8_t* kb = p.k_cache + j * 16;
    const uint8_t* vb = p.v_cache + j * 16;
#pragma unroll
    for (int w = 0; w < TTC / 32; ++w) {
#pragma unroll
      for (int cb = 0; cb < NCH; ++cb) {
#pragma unroll 2
        for (int i = 0; i < 8; ++i) {
          const int src = 4 * i + rq;  // stage row w * 32 + src
          const int y = __shfl_sync(0xffffffffu, yv[w], src);
          if ((mask[w] >> src) & 1u) {
            const int c = cb * TTC + w * 32 + src;  // chunk row
            const uint32_t off = (uint32_t)c * 128u + (uint32_t)((j ^ (c & 7)) << 4);
            const size_t g = (size_t)y * kRowBytes + (size_t)cb * 128;
            cp_async16(kst + off, kb + g);
            cp_async16(vst + off, vb + g);
          }
        }
      }
    }
    if (p.scale_mode == kScalePerToken) {
      const uint32_t sc = kst + (uint32_t)p.off_scale;
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) {
        const int row = rr * 32 + lane;
        if (row < TTC && ((mask[rr] >> lane) & 1u)) {
          cp_async4(sc + row * 4, p.k_scale + yv[rr]);
          cp_async4(sc + TTC * 4 + row * 4, p.v_scale + yv[rr]);
        }
      }
    }
  }

  __device__ __forceinline__ void emit_sparse(StageHdr h) {
    int s;
    if (!acquire_stage(s)) return;
    const int TT = p.TT;
    const uint32_t kst = sm.stage(s, p);
    const uint32_t vst = kst + (uint32_t)TT * (uint32_t)ROWB * NCH;
    const bool empty = !(h.t1 > h.t0);
    int idx[4], phys[4];
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) idx[rr] = phys[rr] = -1;
    if (!empty) {
      if (la_b == h.b && la_pos == h.tbase) {
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) {
          idx[rr] = la_idx[rr];
          phys[rr] = la_phys[rr];
        }
      } else {
        if (nx_b == h.b && nx_pos == h.tbase) {
#pragma unroll
          for (int rr = 0; rr < 4; ++rr) idx[rr] = nx_idx[rr];
        } else {
          load_indices(h.b, h.tbase, p.topk, idx);
        }
        load_phys(h.b, h.L, idx, phys);
      }
      // positions past the stage's range carry no token
#pragma unroll
      for (int rr = 0; rr < 4; ++rr)
        if (h.tbase + rr * 32 + lane >= h.t1) idx[rr] = -1;
    }
    int yv[4];
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const int t = empty ? -1 : idx[rr];
      const bool valid = t >= 0 && t < h.L;
      int y = 0;
      if (valid) {
        int ph = phys[rr];
        if (ph < 0 || ph >= p.num_pages) {
          flag_status(p, kStatusBadPage);
          ph = 0;
        }
        y = (ph * p.Hkv + h.g) * p.S + t % p.S;
      }
      yv[rr] = y;
      h.mask[rr] = __ballot_sync(0xffffffffu, valid);
    }
    __syncwarp();
    if (lane == 0) *sm.hdr(s, p) = h;
    if (!empty) gather_rows(kst, vst, yv, h.mask);
    // The stage is full once lane 0 has published the header and every
    // lane's copies have landed (one noinc arrival per lane).
    __syncwarp();
    if (lane == 0) mbar_arrive(sm.full(s, p));
    cp_async_arrive(sm.full(s, p));
    // look ahead: page ids of the next stage, indices of the one after
    la_b = -1;
    const int next = h.tbase + TT;
    if (!empty && next < p.topk) {
      if (nx_b == h.b && nx_pos == next) {
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) la_idx[rr] = nx_idx[rr];
      } else {
        load_indices(h.b, next, p.topk, la_idx);
      }
      load_phys(h.b, h.L, la_idx, la_phys);
      la_b = h.b;
      la_pos = next;
      nx_b = -1;
      if (next + TT < p.topk) request_indices(h.b, next + TT);
    }
  }

  // Query rows of unit (b, g) into Q ring slot nq % NQ: one bulk copy per
  // query position, since the G heads that share KV head g are contiguous.
  int nq = 0;
  __device__ __forceinline__ bool load_q(int b, int g) {
    const int qs = nq % p.NQ;
    bool got = mbar_wait(sm.qempty(qs, p), ((nq / p.NQ) & 1) ^ 1);
    got = __all_sync(0xffffffffu, got);
    if (!got) {
      ok = false;
      if (lane == 0) {
        flag_status(p, kStatusTimeout);
        sm.misc(p)[0] = 1;
      }
      return false;
    }
    const uint32_t rowb = (uint32_t)p.G * (uint32_t)p.D * 2u;
    if (lane == 0) mbar_arrive_tx(sm.qfull(qs, p), rowb * (uint32_t)p.QL);
    __syncwarp();
    for (int i = lane; i < p.QL; i += 32)
      bulk_load(sm.qbuf(qs, p) + (uint32_t)i * rowb, p.q + ((size_t)(b * p.QL + i) * p.Hq + (size_t)g * p.G) * p.D,
                rowb, sm.qfull(qs, p));
    ++nq;
    return true;
  }

  __device__ __forceinline__ void emit_end() {
    int s;
    if (!acquire_stage(s)) return;
    if (lane == 0) {
      sm.hdr(s, p)->kind_flags = kEnd;
      mbar_arrive(sm.full(s, p));
    }
    if (p.topk > 0) mbar_arrive(sm.full(s, p));  // sparse stages count one arrival per lane too
    __syncwarp();
    ++n;
  }

  // Emit the stages of one segment: chunks [k0, k1) of unit (b, g).
  __device__ __forceinline__ void segment(int b, int g, const UnitRange& r, int k0, int k1, bool whole, int slot, const MergeDesc& md) {
    StageHdr h;
    h.unit = b * p.Hkv + g;
    h.b = b;
    h.g = g;
    h.L = r.L;
    h.mask[0] = h.mask[1] = h.mask[2] = h.mask[3] = 0u;
    h.slot = slot;
    h.nseg = md.nseg;
    h.s0 = md.s0;
    h.sbase = md.sbase;
    h.sstride = md.sstride;
    const int kend = (k1 > k0) ? k1 : k0 + 1;
    if (p.topk == 0 && k1 > k0) {
      // start the first stage's page-id load before the query copy
      const int tbase = (r.c_lo + k0) * p.TT;
      const int lp0 = p.S >= p.TT ? tbase / p.S : max(tbase, r.lo) / p.S;
      stage_window(b, r.L, lp0, p.S < p.TT ? p.TT / p.S : 1);
    } else if (p.topk > 0 && k1 > k0 && !(la_b == b && la_pos == k0 * p.TT) && !(nx_b == b && nx_pos == k0 * p.TT)) {
      request_indices(b, k0 * p.TT);  // the first stage's indices, before the query copy
    }
    if (!load_q(b, g)) return;
    for (int k = k0; k < kend && ok; ++k) {
      h.kind_flags = (k == k0 ? kSegFirst : 0) | (k == kend - 1 ? kSegLast : 0) | (whole ? kSegWhole : 0);
      if (k1 > k0) {
        h.tbase = (r.c_lo + k) * p.TT;
        h.t0 = max(h.tbase, r.lo);
        h.t1 = min(h.tbase + p.TT, r.hi);
      } else {
        h.tbase = 0;
        h.t0 = h.t1 = 0;
      }
      if (p.topk > 0)
        emit_sparse(h);
      else
        emit_dense(h);
      if (!ok) return;
      ++n;
    }
  }

  __device__ __forceinline__ void run() {
    if (lane == 0) {
      prefetch_tmap(tmK);
      prefetch_tmap(tmV);
    }
    if (p.sched == kSchedPerUnit) {
      const int u = blockIdx.x / p.P, j = blockIdx.x % p.P;
      const int b = u / p.Hkv, g = u % p.Hkv;
      const UnitRange r = unit_range(p, b);
      const int k0 = (int)((long long)j * r.n / p.P), k1 = (int)((long long)(j + 1) * r.n / p.P);
      MergeDesc md{p.P, u * p.P, u * p.P, 1};
      segment(b, g, r, k0, k1, p.P == 1, u * p.P + j, md);
    } else {
      // With fewer chunks than CTAs only the first N CTAs take work, so every
      // CTA between a unit's first and last owner holds part of that unit.
      long long N;
      long long cnt_reg[kScanRegs];
      // Sparse units all weigh the same (ceil(topk / TT) chunks whatever the
      // context length): the schedule is closed-form, no length scan.
      const bool uniform = p.topk > 0;
      const long long wu_uniform = (long long)(max(1, (p.topk + p.TT - 1) / p.TT) + p.seg_cost);
      const bool in_regs = !uniform && p.B <= 32 * kScanRegs;
      if (uniform) {
        N = (long long)p.B * p.Hkv * wu_uniform;
      } else if (in_regs) {
        // chunk counts of sequences lane, lane + 32, ... loaded in one round trip
#pragma unroll
        for (int i = 0; i < kScanRegs; ++i) {
          const int b = i * 32 + lane;
          cnt_reg[i] = b < p.B ? seq_weight(p, b) : 0;
        }
        long long t = 0;
#pragma unroll
        for (int i = 0; i < kScanRegs; ++i) t += cnt_reg[i];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
        N = t;
      } else {
        N = balanced_total(p, lane);
      }
      const long long C = min((long long)p.C, N);
      const long long c = blockIdx.x;
      long long x = c < C ? sched_start(c, N, C) : 0;
      const long long x1 = c < C ? sched_start(c + 1, N, C) : 0;
      // sequence holding global chunk xx and the chunk count before it
      auto locate = [&](long long xx, int& b, long long& excl) {
        if (uniform) {
          b = (int)(xx / ((long long)p.Hkv * wu_uniform));
          excl = (long long)b * p.Hkv * wu_uniform;
        } else if (in_regs) {
          long long base = 0;
          b = p.B;
          excl = 0;
#pragma unroll
          for (int i = 0; i < kScanRegs; ++i) {
            if (i * 32 >= p.B) break;
            long long incl = cnt_reg[i];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
              const long long v = __shfl_up_sync(0xffffffffu, incl, off);
              if (lane >= off) incl += v;
            }
            const long long total = __shfl_sync(0xffffffffu, incl, 31);
            const unsigned hit = __ballot_sync(0xffffffffu, base + incl > xx);
            if (hit && b == p.B) {
              const int first = __ffs(hit) - 1;
              b = i * 32 + first;
              excl = base + __shfl_sync(0xffffffffu, incl - cnt_reg[i], first);
            }
            base += total;
          }
        } else {
          balanced_find(p, lane, xx, b, excl);
        }
      };
      if (x < x1) {
        int b;
        long long excl;
        locate(x, b, excl);
        UnitRange r = unit_range(p, b);
        long long nb = max(1, r.n), wu = nb + p.seg_cost;
        int g = (int)((x - excl) / wu);
        while (x < x1 && ok) {
          const long long Pu = excl + g * wu, R0 = Pu + p.seg_cost;
          const long long lo = max(x, R0), hi = min(x1, R0 + nb);
          if (lo < hi) {
            // A unit split over CTAs c1..c2 writes one partial per CTA: slot
            // 2c for the unit CTA c starts with, 2c + 1 for the one it ends
            // with (a unit one CTA covers alone is written as output directly).
            const MergeDesc md = balanced_desc(Pu, nb, p.seg_cost, N, C);
            const int slot = (int)(2 * c + ((c == sched_owner(R0, N, C) && sched_start(c, N, C) < Pu) ? 1 : 0));
            if (r.n > 0)
              segment(b, g, r, (int)(lo - R0), (int)(hi - R0), md.nseg == 1, slot, md);
            else
              segment(b, g, r, 0, 0, md.nseg == 1, slot, md);
          }
          x = Pu + wu;
          if (++g == p.Hkv) {
            g = 0;
            excl += (long long)p.Hkv * wu;
            ++b;
            if (b < p.B) {
              r = unit_range(p, b);
              nb = max(1, r.n);
              wu = nb + p.seg_cost;
            }
          }
        }
      }
    }
    if (ok) emit_end();
    if (!ok) {
      // Wait (bounded) for copies this warp issued that may still be in flight.
      if (p.topk > 0) cp_async_wait_all();
      const int first = max(0, n - p.NS);
      for (int m = first; m < n; ++m) (void)mbar_wait(sm.full(m % p.NS, p), (m / p.NS) & 1);
      for (int m = max(0, nq - p.NQ); m < nq; ++m) (void)mbar_wait(sm.qfull(m % p.NQ, p), (m / p.NQ) & 1);
    }
  }
};

// ------------------------------------------------------------ unit merges
// Count one partial of a split unit; the last of its nseg partials queues
// the unit's merge for this CTA (thread 0 only).
__device__ __forceinline__ void la_arrive(const PaParams& p, Smem sm, int b, int g, int unit, const MergeDesc& md) {
  int* cnt = p.counters + (size_t)unit * kCounterStride;
  const int prev = atomicAdd(cnt, 1);
  if (prev != md.nseg - 1) return;
  atomicExch(cnt, 0);
  volatile int* npend = sm.misc(p) + 2;
  const int idx = *npend;
  int4* q = reinterpret_cast<int4*>(sm.base + p.off_pend) + 2 * idx;
  q[0] = make_int4(b, g, unit, md.nseg);
  q[1] = make_int4(md.s0, md.sbase, md.sstride, 0);
  *npend = idx + 1;
}

// Run and clear the queued merges with the nthr consumer threads (named
// barrier 1).
template <int D>
__device__ void la_run_queue(const PaParams& p, Smem sm, float vscale, int nthr) {
  const int cnt = *(sm.misc(p) + 2);
  if (cnt == 0) return;
  __threadfence();
  for (int i = 0; i < cnt; ++i) {
    const int4* q = reinterpret_cast<const int4*>(sm.base + p.off_pend) + 2 * i;
    const int4 a = q[0], c = q[1];
    const MergeDesc md{a.w, c.x, c.y, c.z};
    merge_elems<D>(
        p, vscale, md.nseg, a.x, a.y, threadIdx.x, nthr, 0, p.R * (D / 4),
        [&](int k, int r) {
          return __ldcg(reinterpret_cast<const float2*>(p.part_ml + ((size_t)merge_slot(md, k) * p.Rpad + r) * 2));
        },
        [&](int k, int r, int d) {
          return __ldcg(
              reinterpret_cast<const float4*>(p.part_o + ((size_t)merge_slot(md, k) * p.Rpad + r) * D + d));
        });
  }
  named_bar(1, nthr);
  if (threadIdx.x == 0) *(sm.misc(p) + 2) = 0;
  named_bar(1, nthr);
}

// Cluster merge: CTA `rank` merges its share of the unit's output elements
// from the partials of all P CTAs (partition order), read over distributed
// shared memory.
template <int D>
__device__ void cluster_merge_unit(const PaParams& p, Smem sm, float vscale, int unit, int tid, int nthr) {
  const int b = unit / p.Hkv, g = unit % p.Hkv;
  uint32_t rank;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
  const int E = p.R * (D / 4);
  const int e0 = (int)((long long)rank * E / p.P), e1 = (int)((long long)(rank + 1) * E / p.P);
  const uint32_t cp_local = sm.base_u32 + p.off_cpart;
  const uint32_t ml_off = (uint32_t)p.Rpad * D * 4u;
  merge_elems<D>(
      p, vscale, p.P, b, g, tid, nthr, e0, e1,
      [&](int k, int r) {
        uint32_t remote;
        asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(cp_local + ml_off + 8u * r), "r"(k));
        float2 v;
        asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(remote));
        return v;
      },
      [&](int k, int r, int d) {
        uint32_t remote;
        asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                     : "=r"(remote)
                     : "r"(cp_local + 4u * (uint32_t)(r * D + d)), "r"(k));
        float4 v;
        asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                     : "r"(remote));
        return v;
      });
}

// ================================================================ consumers
// Per-stage header fields every consumer warp needs. The sparse validity
// words are separate scalars (selected by comparison, never indexed with a
// runtime value) so that the whole view stays in registers.
struct StageView {
  int flags, tbase, t0, t1, L, unit, b, g;
  unsigned m0, m1, m2, m3;
  __device__ __forceinline__ unsigned mask_word(int w) const {
    return w == 0 ? m0 : (w == 1 ? m1 : (w == 2 ? m2 : m3));
  }
};

// QF16 (BF16 caches only): the queries are FP16; each is split exactly into
// BF16 hi + lo (an FP16 value's 11 significant bits leave at most 4 for lo)
// and S takes one BF16 MMA per term. FP8 caches convert any query type to
// FP16 operands at the segment start (a runtime flag).
// FP4: MXFP4 caches (head_dim 128, with FP8 = VTOK = true: FP16 queries, P and
// V; the per-token K and V factors come from the block scales).
// TV: BF16 V in the transposed layout (chunks of 8 tokens per head dim).
template <bool FP8, int D, int NT, bool VTOK, int TW, bool QF16 = false, bool FP4 = false, bool TV = false>
struct Consumer {
  static_assert(!FP4 || (FP8 && VTOK && D == 128), "MXFP4 runs the FP8 per-token path at head_dim 128");
  static_assert(!TV || !FP8, "transposed V: BF16 caches");
  static constexpr int ELT = FP8 ? 1 : 2;
  static constexpr int NCH = FP4 ? 1 : D * ELT / 128;  // column blocks per token row
  static constexpr uint32_t ROWB = FP4 ? 64u : 128u;   // bytes of a stage row per block
  static constexpr uint32_t TILEB = 16u * ROWB;        // bytes of a 16-token tile per block
  static constexpr int KSTEPS = D / 16;
  static constexpr int MT = D / 16;
  static constexpr int KS_BLK = KSTEPS / NCH;
  static constexpr int MT_BLK = MT / NCH;
  static constexpr bool PV_F16 = FP8;  // FP8 caches: FP16 P and V; BF16 caches: BF16 P
  static constexpr int RW = 8 * NT;
  static constexpr int DPB = 128 / ELT;  // head dims per 128-byte block

  const PaParams& p;
  Smem sm;
  int lane, g4, t4, wr, wt;
  uint32_t koff[NCH][2][2];  // [block][token g4 / g4+8][chunk half], tile-relative
  uint32_t voff[NCH][4];     // [block][token 2t4, 2t4+1, 2t4+8, 2t4+9]
  // MXFP4: K chunk t4 (32 dims = one MX block) of tokens g4 / g4+8; V bytes
  // [8 g4, 8 g4 + 8) (dims [16 g4, 16 g4 + 16), MX block g4 / 2) of tokens
  // 2t4, 2t4+1, 2t4+8, 2t4+9 (64-byte rows, 64-byte swizzle)
  uint32_t koff4[2], voff4[4];
  // transposed V: a stage chunk of 8 tokens is D/8 rows of 128 bytes (8 dims
  // x 8 tokens) under the 128-byte swizzle; the A fragment of m-tile mt of a
  // 64-dim block holds dims 8 g4 + 2 mt (row g4) and + 1 (row g4 + 8), the
  // plain layout's order, read as 4 bytes (tokens 2 t4, 2 t4 + 1) at
  // row g4, chunk (2 mt + h) ^ g4
  uint32_t tvoff[4][2];
  float kscale = 1.f, vscale = 1.f;
  // per segment
  uint32_t qf[NT][KSTEPS][2];
  uint32_t qlo[QF16 ? NT : 1][QF16 ? KSTEPS : 1][2];  // FP16 queries on BF16 caches: the lo terms
  float crow[NT][2];
  int prow[NT][2];  // query position of the thread's two rows per n-tile
  float mrun[NT][2], lrun[NT][2];
  float o[MT][NT][4];
  // Per-token V scales: O is kept in units of 2^vexp so that P * v_scale / 2^vexp
  // stays <= 1 and is rounded to FP16 (exact power-of-two rescales of O).
  int vexp = -127;

  __device__ Consumer(const PaParams& p_, Smem s) : p(p_), sm(s) {
    lane = threadIdx.x & 31;
    g4 = lane >> 2;
    t4 = lane & 3;
    const int cw = threadIdx.x >> 5;
    wr = cw % p.Wr;
    wt = cw / p.Wr;
    if (FP8 && p.scale_mode == kScalePerTensor) kscale = __ldg(p.k_scale);
    vscale = per_tensor_vscale(p);
    // Swizzled shared-memory offsets: row r's 16-byte chunk c sits at chunk
    // c ^ (r & 7) (128-byte swizzle, dense and sparse stages alike).
#pragma unroll
    for (int cb = 0; cb < NCH; ++cb) {
#pragma unroll
      for (int ab = 0; ab < 2; ++ab) {
        const int row = g4 + 8 * ab;
#pragma unroll
        for (int hl = 0; hl < 2; ++hl)
          koff[cb][ab][hl] = (uint32_t)(cb * p.TT + row) * 128u + (uint32_t)(((2 * t4 + hl) ^ (row & 7)) << 4);
      }
      const int vr[4] = {2 * t4, 2 * t4 + 1, 2 * t4 + 8, 2 * t4 + 9};
#pragma unroll
      for (int k = 0; k < 4; ++k)
        voff[cb][k] = (uint32_t)(cb * p.TT + vr[k]) * 128u + (uint32_t)((g4 ^ (vr[k] & 7)) << 4);
    }
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
        tvoff[mt][hh] = (uint32_t)g4 * 128u + (uint32_t)(((2 * mt + hh) ^ g4) << 4) + 4u * (uint32_t)t4;
    // 64-byte swizzle: row r's 16-byte chunk c sits at chunk c ^ ((r >> 1) & 3)
#pragma unroll
    for (int ab = 0; ab < 2; ++ab) {
      const int row = g4 + 8 * ab;
      koff4[ab] = (uint32_t)row * 64u + (uint32_t)((t4 ^ ((row >> 1) & 3)) << 4);
    }
    {
      const int vr[4] = {2 * t4, 2 * t4 + 1, 2 * t4 + 8, 2 * t4 + 9};
#pragma unroll
      for (int k = 0; k < 4; ++k)
        voff4[k] = (uint32_t)vr[k] * 64u + (uint32_t)((((g4 >> 1) ^ ((vr[k] >> 1) & 3)) << 4) | ((g4 & 1) << 3));
    }
  }

  __device__ __forceinline__ int row_of(int j, int rho) const { return wr * RW + 8 * j + 2 * t4 + rho; }

  // XOR on the float4 column of row r in the token-group merge buffer. One
  // 128-bit store instruction covers lanes t4 = 0..3 (rows 2*t4 + rho) and two
  // g4 values; the XOR sends those eight lanes to eight different 16-byte
  // bank groups. Readers walk a row's columns in order, so they stay
  // conflict-free under any XOR below 8.
  __device__ __forceinline__ static int merge_swz(int r) {
    const int t = (r >> 1) & 3;
    return ELT == 1 ? t : ((t & 1) | ((t & 2) << 1));
  }

  int nq = 0;  // segments begun (Q ring position)

  // Start a segment of unit (b, g): take its query rows from the Q ring.
  // Returns false if the rows did not arrive in time.
  __device__ bool begin_segment(int L) {
    const int qs = nq % p.NQ;
    bool got = mbar_wait(sm.qfull(qs, p), (nq / p.NQ) & 1);
    got = __all_sync(0xffffffffu, got);
    if (!got) return false;
    ++nq;
    // Q rows of this warp's slice as MMA B fragments (row n = g4), with the
    // head-dim permutation that matches how K rows are read from shared memory.
    // Slot rows are laid out like the unit's rows of q: row r = i * G + head.
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const int r = wr * RW + 8 * j + g4;
      const bool valid = r < p.R;
      const uint32_t qrow = sm.qbuf(qs, p) + (uint32_t)(valid ? r : 0) * (uint32_t)(D * 2);
      float crow_n = 0.f;
      if constexpr (FP8) {
        // 32 values per block: d in [cb*128 + 32*t4, +32)
        const bool qh = p.q_f16 != 0;
        float amax = 0.f;
        uint4 raw[NCH][4];
#pragma unroll
        for (int cb = 0; cb < NCH; ++cb)
#pragma unroll
          for (int v = 0; v < 4; ++v)
            raw[cb][v] = valid ? lds128(qrow + (uint32_t)(cb * 128 + 32 * t4) * 2u + 16u * v) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int cb = 0; cb < NCH; ++cb)
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const uint32_t w[4] = {raw[cb][v].x, raw[cb][v].y, raw[cb][v].z, raw[cb][v].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              amax = fmaxf(amax, fabsf(q_bits_to_f32(w[e] & 0xFFFFu, qh)));
              amax = fmaxf(amax, fabsf(q_bits_to_f32(w[e] >> 16, qh)));
            }
          }
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        // power-of-two row scale: amax * 2^e in [2^14, 2^15) keeps every
        // BF16 value exact in FP16 apart from far-below-max tails
        int e = 0;
        if (amax > 0.f) {
          const int ex = (int)((__float_as_uint(amax) >> 23) & 0xFF) - 127;
          e = max(-126, min(126, 14 - ex));
        }
        const float sc = __uint_as_float((uint32_t)(e + 127) << 23);
        const float inv = __uint_as_float((uint32_t)(127 - e) << 23);
#pragma unroll
        for (int cb = 0; cb < NCH; ++cb)
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const uint32_t w[4] = {raw[cb][v].x, raw[cb][v].y, raw[cb][v].z, raw[cb][v].w};
            // words w[0..3] hold d = 32*t4 + 8v + {0..7}; k-step 2v + hw takes 4 of them
#pragma unroll
            for (int hw = 0; hw < 2; ++hw) {
              const int s = cb * KS_BLK + 2 * v + hw;
              qf[j][s][0] =
                  pack_f16(q_bits_to_f32(w[2 * hw] & 0xFFFFu, qh) * sc, q_bits_to_f32(w[2 * hw] >> 16, qh) * sc);
              qf[j][s][1] = pack_f16(q_bits_to_f32(w[2 * hw + 1] & 0xFFFFu, qh) * sc,
                                     q_bits_to_f32(w[2 * hw + 1] >> 16, qh) * sc);
            }
          }
        crow_n = valid ? inv * p.sm_scale_log2 * (p.scale_mode == kScalePerTensor ? kscale : 1.f) : 0.f;
      } else {
        // 16 values per block: d in [cb*64 + 16*t4, +16)
#pragma unroll
        for (int cb = 0; cb < NCH; ++cb)
#pragma unroll
          for (int v = 0; v < 2; ++v) {
            const uint4 w = valid ? lds128(qrow + (uint32_t)(cb * 64 + 16 * t4) * 2u + 16u * v) : make_uint4(0, 0, 0, 0);
            const int s0 = cb * KS_BLK + 2 * v;
            if constexpr (QF16) {
              const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float a = f16_bits_to_f32(ww[e] & 0xFFFFu), b = f16_bits_to_f32(ww[e] >> 16);
                const uint32_t hi = pack_bf16(a, b);
                const uint32_t lo = pack_bf16(a - bf16_bits_to_f32(hi & 0xFFFFu), b - bf16_bits_to_f32(hi >> 16));
                qf[j][s0 + e / 2][e & 1] = hi;
                qlo[j][s0 + e / 2][e & 1] = lo;
              }
            } else {
              qf[j][s0][0] = w.x;
              qf[j][s0][1] = w.y;
              qf[j][s0 + 1][0] = w.z;
              qf[j][s0 + 1][1] = w.w;
            }
          }
        crow_n = valid ? p.sm_scale_log2 : 0.f;
      }
#pragma unroll
      for (int rho = 0; rho < 2; ++rho) {
        crow[j][rho] = __shfl_sync(0xffffffffu, crow_n, (2 * t4 + rho) * 4);
        const int rr = row_of(j, rho);
        prow[j][rho] = (rr < p.R) ? (L - p.QL + rr / p.G) : -(1 << 30);
        mrun[j][rho] = -INFINITY;
        lrun[j][rho] = 0.f;
      }
    }
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[mt][j][e] = 0.f;
    vexp = -127;
    __syncwarp();  // every lane has read its rows
    if (lane == 0) mbar_arrive(sm.qempty(qs, p));
    return true;
  }

  // Does stage row `row` carry a real token (one that some query row may see)?
  __device__ __forceinline__ bool token_ok(const StageView& h, int row) const {
    if (p.topk > 0) return ((h.mask_word(row >> 5) >> (row & 31)) & 1u) != 0u;
    const int t = h.tbase + row;
    return t >= h.t0 && t < h.t1;
  }
  __device__ __forceinline__ bool score_ok(const StageView& h, int row, int j, int rho) const {
    if (!token_ok(h, row)) return false;
    const int pr = prow[j][rho];
    if (p.topk > 0) return pr > -(1 << 29);
    const int t = h.tbase + row;
    bool ok = pr > -(1 << 29);
    if (p.causal) ok = ok && t <= pr;
    if (p.window > 0) ok = ok && t > pr - p.window;
    return ok;
  }

  // One warp step: TW consecutive 16-token tiles starting at tile tau0.
  __device__ void step(const StageView& h, uint32_t kst, uint32_t vst, uint32_t sst, int tau0) {
    bool interior[TW];
    bool any = false;
#pragma unroll
    for (int u = 0; u < TW; ++u) {
      const int tau = tau0 + u;
      bool live;
      if (p.topk > 0) {
        const unsigned m16 = (h.mask_word(tau >> 1) >> (16 * (tau & 1))) & 0xFFFFu;
        live = m16 != 0u;
        interior[u] = m16 == 0xFFFFu;
      } else {
        const int ta = h.tbase + 16 * tau;
        live = !(ta >= h.t1 || ta + 16 <= h.t0);
        const int lo_all = p.window > 0 ? max(0, h.L - p.window) : 0;
        const int hi_all = p.causal ? h.L - p.QL + 1 : h.L;
        interior[u] = ta >= max(h.t0, lo_all) && ta + 16 <= min(h.t1, hi_all);
      }
      any |= live;
    }
    if (!any) return;
    // ---- S^T = K Q^T for each tile ------------------------------------------
    float sacc[TW][NT][4];
#pragma unroll
    for (int u = 0; u < TW; ++u)
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[u][j][e] = 0.f;
    float ks4[TW][2];  // MXFP4: the K rows' factors 2^(largest block code - 127)
    if constexpr (FP4) {
#pragma unroll
      for (int u = 0; u < TW; ++u) {
        const uint32_t tb = kst + (uint32_t)(tau0 + u) * TILEB;
        const int rA = 16 * (tau0 + u) + g4;
        const uint32_t swa = lds32(sst + (uint32_t)rA * 4u), swb = lds32(sst + (uint32_t)(rA + 8) * 4u);
        ks4[u][0] = e8m0_to_f32(mx_max_code(swa));
        ks4[u][1] = e8m0_to_f32(mx_max_code(swb));
        const uint32_t fa = mx_block_factor(swa, t4), fb = mx_block_factor(swb, t4);
        const uint4 ka = lds128(tb + koff4[0]), kb = lds128(tb + koff4[1]);
        const uint32_t wa[4] = {ka.x, ka.y, ka.z, ka.w};
        const uint32_t wb[4] = {kb.x, kb.y, kb.z, kb.w};
#pragma unroll
        for (int s = 0; s < KSTEPS; ++s) {
          // k-step s: dims 32 t4 + 4 s + {0, 1} (byte 2 s) and + {2, 3} (byte 2 s + 1)
          const uint32_t xa = wa[s >> 1] >> (16 * (s & 1)), xb = wb[s >> 1] >> (16 * (s & 1));
          const uint32_t a0 = mul_f16x2(e2m1x2_to_f16x2(xa), fa), a2 = mul_f16x2(e2m1x2_to_f16x2(xa >> 8), fa);
          const uint32_t a1 = mul_f16x2(e2m1x2_to_f16x2(xb), fb), a3 = mul_f16x2(e2m1x2_to_f16x2(xb >> 8), fb);
#pragma unroll
          for (int j = 0; j < NT; ++j) mma16816<true>(sacc[u][j], a0, a1, a2, a3, qf[j][s][0], qf[j][s][1]);
        }
      }
    }
#pragma unroll
    for (int cb = 0; cb < (FP4 ? 0 : NCH); ++cb) {
#pragma unroll
      for (int hl = 0; hl < 2; ++hl) {
        uint4 ka[TW], kb[TW];
#pragma unroll
        for (int u = 0; u < TW; ++u) {
          const uint32_t tb = kst + (uint32_t)(tau0 + u) * TILEB;
          ka[u] = lds128(tb + koff[cb][0][hl]);
          kb[u] = lds128(tb + koff[cb][1][hl]);
        }
#pragma unroll
        for (int u = 0; u < TW; ++u) {
          const uint32_t wa[4] = {ka[u].x, ka[u].y, ka[u].z, ka[u].w};
          const uint32_t wb[4] = {kb[u].x, kb[u].y, kb[u].z, kb[u].w};
          if constexpr (FP8) {
#pragma unroll
            for (int w = 0; w < 4; ++w) {
              const int s = cb * KS_BLK + hl * 4 + w;
              const uint32_t a0 = e4m3x2_to_f16x2(wa[w]), a2 = e4m3x2_to_f16x2(wa[w] >> 16);
              const uint32_t a1 = e4m3x2_to_f16x2(wb[w]), a3 = e4m3x2_to_f16x2(wb[w] >> 16);
#pragma unroll
              for (int j = 0; j < NT; ++j) mma16816<true>(sacc[u][j], a0, a1, a2, a3, qf[j][s][0], qf[j][s][1]);
            }
          } else {
#pragma unroll
            for (int w2 = 0; w2 < 2; ++w2) {
              const int s = cb * KS_BLK + hl * 2 + w2;
#pragma unroll
              for (int j = 0; j < NT; ++j)
                mma16816<false>(sacc[u][j], wa[2 * w2], wb[2 * w2], wa[2 * w2 + 1], wb[2 * w2 + 1], qf[j][s][0],
                                qf[j][s][1]);
              if constexpr (QF16) {
#pragma unroll
                for (int j = 0; j < NT; ++j)
                  mma16816<false>(sacc[u][j], wa[2 * w2], wb[2 * w2], wa[2 * w2 + 1], wb[2 * w2 + 1], qlo[j][s][0],
                                  qlo[j][s][1]);
              }
            }
          }
        }
      }
    }
    // ---- scale (before masking), mask, online softmax over the TW tiles -----
    const bool ktok = FP8 && p.scale_mode == kScalePerToken;
    float ks[TW][2], vs[TW][2];
#pragma unroll
    for (int u = 0; u < TW; ++u) {
      const int rA = 16 * (tau0 + u) + g4;
      ks[u][0] = ks[u][1] = vs[u][0] = vs[u][1] = 1.f;
      if constexpr (FP4) {
        ks[u][0] = ks4[u][0];
        ks[u][1] = ks4[u][1];
        vs[u][0] = e8m0_to_f32(mx_max_code(lds32(sst + (uint32_t)(p.TT + rA) * 4u)));
        vs[u][1] = e8m0_to_f32(mx_max_code(lds32(sst + (uint32_t)(p.TT + rA + 8) * 4u)));
      } else if (ktok) {
        ks[u][0] = lds_f32(sst + rA * 4);
        ks[u][1] = lds_f32(sst + (rA + 8) * 4);
      }
      if constexpr (VTOK && !FP4) {
        vs[u][0] = lds_f32(sst + p.TT * 4 + rA * 4);
        vs[u][1] = lds_f32(sst + p.TT * 4 + (rA + 8) * 4);
      }
    }
    bool rescale = false;
    float vfix = 1.f;
    if constexpr (VTOK) {
      // the step's largest valid V scale sets the power-of-two unit of O
      float vm = 0.f;
#pragma unroll
      for (int u = 0; u < TW; ++u) {
        const int rA = 16 * (tau0 + u) + g4;
        vm = fmaxf(vm, (interior[u] || token_ok(h, rA)) ? vs[u][0] : 0.f);
        vm = fmaxf(vm, (interior[u] || token_ok(h, rA + 8)) ? vs[u][1] : 0.f);
      }
      vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, 4));
      vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, 8));
      vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, 16));
      if (vm > 0.f) {
        const int et = min(120, (int)((__float_as_uint(vm) >> 23) & 0xFF) - 126);  // vm < 2^et
        if (et > vexp) {
          vfix = vexp <= -127 ? 0.f : __uint_as_float((uint32_t)max(0, vexp - et + 127) << 23);
          vexp = et;
          rescale = true;
        }
      }
      const float inv = __uint_as_float((uint32_t)(127 - max(vexp, -126)) << 23);
#pragma unroll
      for (int u = 0; u < TW; ++u) {
        vs[u][0] *= inv;
        vs[u][1] *= inv;
      }
    }
    uint32_t pb[TW][NT][2];
    float alpha[NT][2];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      float x[TW][4];
#pragma unroll
      for (int u = 0; u < TW; ++u) {
#pragma unroll
        for (int e = 0; e < 4; ++e) x[u][e] = sacc[u][j][e] * crow[j][e & 1] * ks[u][e >> 1];
        if (!interior[u]) {
          const int rA = 16 * (tau0 + u) + g4;
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (!score_ok(h, e < 2 ? rA : rA + 8, j, e & 1)) x[u][e] = -INFINITY;
        }
      }
      float pe[TW][4];
#pragma unroll
      for (int rho = 0; rho < 2; ++rho) {
        float mx = -INFINITY;
#pragma unroll
        for (int u = 0; u < TW; ++u) mx = fmaxf(mx, fmaxf(x[u][rho], x[u][rho + 2]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const float mnew = fmaxf(mrun[j][rho], mx);
        const float muse = (mnew == -INFINITY) ? 0.f : mnew;
        const float a = ex2(mrun[j][rho] - muse);
        float sum = 0.f;
#pragma unroll
        for (int u = 0; u < TW; ++u) {
          pe[u][rho] = ex2(x[u][rho] - muse);
          pe[u][rho + 2] = ex2(x[u][rho + 2] - muse);
          sum += pe[u][rho] + pe[u][rho + 2];
        }
        lrun[j][rho] = lrun[j][rho] * a + sum;
        mrun[j][rho] = mnew;
        alpha[j][rho] = a * vfix;
        rescale |= (a != 1.f);
      }
#pragma unroll
      for (int u = 0; u < TW; ++u) {
        if constexpr (VTOK) {
          // per-token V scale folded into P before rounding (masked tokens: 0)
          pe[u][0] *= vs[u][0];
          pe[u][1] *= vs[u][0];
          pe[u][2] *= vs[u][1];
          pe[u][3] *= vs[u][1];
          if (!interior[u]) {
            const int rA = 16 * (tau0 + u) + g4;
            if (!token_ok(h, rA)) pe[u][0] = pe[u][1] = 0.f;
            if (!token_ok(h, rA + 8)) pe[u][2] = pe[u][3] = 0.f;
          }
        }
        uint32_t x0, x1;
        if constexpr (PV_F16) {
          x0 = pack_f16(pe[u][0], pe[u][1]);
          x1 = pack_f16(pe[u][2], pe[u][3]);
        } else {
          x0 = pack_bf16(pe[u][0], pe[u][1]);
          x1 = pack_bf16(pe[u][2], pe[u][3]);
        }
        pb[u][j][0] = movm_trans(x0);
        pb[u][j][1] = movm_trans(x1);
      }
    }
    if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          o[mt][j][0] *= alpha[j][0];
          o[mt][j][2] *= alpha[j][0];
          o[mt][j][1] *= alpha[j][1];
          o[mt][j][3] *= alpha[j][1];
        }
    }
    // ---- O^T += V^T P^T ---------------------------------------------------------
#pragma unroll
    for (int u = 0; u < TW; ++u) {
      if constexpr (FP4) {
        // tokens 2t4, 2t4+1, 2t4+8, 2t4+9: dims [16 g4, 16 g4 + 16), byte i = dims 16 g4 + 2i, +1;
        // m-tile mt rows g4 / g4+8 = dims 16 g4 + 2 mt / + 1 (the FP8 head_dim-128 order)
        const uint32_t tb = vst + (uint32_t)(tau0 + u) * TILEB;
        const int vr0 = 16 * (tau0 + u) + 2 * t4;
        const int vrow[4] = {vr0, vr0 + 1, vr0 + 8, vr0 + 9};
        uint2 vv[4];
        uint32_t fv[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          vv[k] = lds64(tb + voff4[k]);
          fv[k] = mx_block_factor(lds32(sst + (uint32_t)(p.TT + vrow[k]) * 4u), g4 >> 1);
        }
        if (!interior[u]) {
#pragma unroll
          for (int k = 0; k < 4; ++k)
            if (!token_ok(h, vrow[k])) vv[k] = make_uint2(0u, 0u);
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          uint32_t w[4];
#pragma unroll
          for (int k = 0; k < 4; ++k)
            w[k] = mul_f16x2(e2m1x2_to_f16x2((mt < 4 ? vv[k].x : vv[k].y) >> (8 * (mt & 3))), fv[k]);
          const uint32_t r0 = __byte_perm(w[0], w[1], 0x5410u), r1 = __byte_perm(w[0], w[1], 0x7632u);
          const uint32_t r2 = __byte_perm(w[2], w[3], 0x5410u), r3 = __byte_perm(w[2], w[3], 0x7632u);
#pragma unroll
          for (int j = 0; j < NT; ++j) mma16816<true>(o[mt][j], r0, r1, r2, r3, pb[u][j][0], pb[u][j][1]);
        }
      }
      if constexpr (TV) {
        static_assert(MT_BLK == 4, "64-dim blocks");
        // tokens 2t4, 2t4+1 (first chunk) and 2t4+8, 2t4+9 (second); those
        // outside the stage's range are zeroed
        const uint32_t tb = vst + (uint32_t)(tau0 + u) * (uint32_t)(32 * D);
        uint32_t m0 = 0xFFFFFFFFu, m1 = 0xFFFFFFFFu;
        if (!interior[u]) {
          const int vr0 = 16 * (tau0 + u) + 2 * t4;
          m0 = (token_ok(h, vr0) ? 0xFFFFu : 0u) | (token_ok(h, vr0 + 1) ? 0xFFFF0000u : 0u);
          m1 = (token_ok(h, vr0 + 8) ? 0xFFFFu : 0u) | (token_ok(h, vr0 + 9) ? 0xFFFF0000u : 0u);
        }
#pragma unroll
        for (int cb = 0; cb < NCH; ++cb)
#pragma unroll
          for (int mt = 0; mt < MT_BLK; ++mt) {
            const uint32_t base = tb + (uint32_t)cb * 1024u;
            const uint32_t r0 = lds32(base + tvoff[mt][0]) & m0;
            const uint32_t r1 = lds32(base + tvoff[mt][1]) & m0;
            const uint32_t r2 = lds32(base + (uint32_t)(16 * D) + tvoff[mt][0]) & m1;
            const uint32_t r3 = lds32(base + (uint32_t)(16 * D) + tvoff[mt][1]) & m1;
#pragma unroll
            for (int j = 0; j < NT; ++j)
              mma16816<false>(o[cb * MT_BLK + mt][j], r0, r1, r2, r3, pb[u][j][0], pb[u][j][1]);
          }
      }
#pragma unroll
      for (int cb = 0; cb < ((FP4 || TV) ? 0 : NCH); ++cb) {
        uint4 vv[4];
        const uint32_t tb = vst + (uint32_t)(tau0 + u) * TILEB;
#pragma unroll
        for (int k = 0; k < 4; ++k) vv[k] = lds128(tb + voff[cb][k]);
        if (!interior[u]) {
          const int vr0 = 16 * (tau0 + u) + 2 * t4;
          const int vrow[4] = {vr0, vr0 + 1, vr0 + 8, vr0 + 9};
#pragma unroll
          for (int k = 0; k < 4; ++k)
            if (!token_ok(h, vrow[k])) vv[k] = make_uint4(0, 0, 0, 0);
        }
        const uint32_t va[4] = {vv[0].x, vv[0].y, vv[0].z, vv[0].w};
        const uint32_t vb[4] = {vv[1].x, vv[1].y, vv[1].z, vv[1].w};
        const uint32_t vc[4] = {vv[2].x, vv[2].y, vv[2].z, vv[2].w};
        const uint32_t vd[4] = {vv[3].x, vv[3].y, vv[3].z, vv[3].w};
        if constexpr (FP8) {
#pragma unroll
          for (int mt = 0; mt < MT_BLK; ++mt) {
            const int wi = mt >> 1;
            const uint32_t sel = (mt & 1) ? 0x7362u : 0x5140u;
            const uint32_t x01 = __byte_perm(va[wi], vb[wi], sel);
            const uint32_t x23 = __byte_perm(vc[wi], vd[wi], sel);
            const uint32_t r0 = e4m3x2_to_f16x2(x01), r1 = e4m3x2_to_f16x2(x01 >> 16);
            const uint32_t r2 = e4m3x2_to_f16x2(x23), r3 = e4m3x2_to_f16x2(x23 >> 16);
#pragma unroll
            for (int j = 0; j < NT; ++j) mma16816<true>(o[cb * MT_BLK + mt][j], r0, r1, r2, r3, pb[u][j][0], pb[u][j][1]);
          }
        } else {
#pragma unroll
          for (int mt = 0; mt < MT_BLK; ++mt) {
            const uint32_t r0 = __byte_perm(va[mt], vb[mt], 0x5410u);
            const uint32_t r1 = __byte_perm(va[mt], vb[mt], 0x7632u);
            const uint32_t r2 = __byte_perm(vc[mt], vd[mt], 0x5410u);
            const uint32_t r3 = __byte_perm(vc[mt], vd[mt], 0x7632u);
#pragma unroll
            for (int j = 0; j < NT; ++j)
              mma16816<false>(o[cb * MT_BLK + mt][j], r0, r1, r2, r3, pb[u][j][0], pb[u][j][1]);
          }
        }
      }
    }
  }

  // ---------------------------------------------------------------- epilogue
  // Segment end. The token-group warps hold partial states of the same rows;
  // they merge them through the segment's last stage buffer (free once every
  // warp has read it) in a fixed order, then write the BF16 output (a unit the
  // CTA covers alone), a global partial (a split unit) or the cluster partial.
  // Only then is the stage handed back to the producer.
  __device__ void end_segment(const StageView& h, int slot, const MergeDesc& md, int s) {
    const bool whole = (h.flags & kSegWhole) != 0;
    const bool cluster = p.merge == kMergeCluster;
    const float ounit = VTOK ? __uint_as_float((uint32_t)(max(vexp, -126) + 127) << 23) : 1.f;
    const int nthr = p.NCW * 32;
    float* cp_o = reinterpret_cast<float*>(sm.base + p.off_cpart);
    float* cp_ml = cp_o + (size_t)p.Rpad * D;
    float lsum[NT][2];
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int rho = 0; rho < 2; ++rho) {
        float l = lrun[j][rho];
        l += __shfl_xor_sync(0xffffffffu, l, 4);
        l += __shfl_xor_sync(0xffffffffu, l, 8);
        l += __shfl_xor_sync(0xffffffffu, l, 16);
        lsum[j][rho] = l;
      }
    if (p.Wt == 1) {
      // one token group: this warp's rows are complete in registers
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.empty(s, p));
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int rho = 0; rho < 2; ++rho) {
          const int r = row_of(j, rho);
          if (r >= p.R) continue;
#pragma unroll
          for (int cb = 0; cb < NCH; ++cb) {
            float v[DPB / 8];
#pragma unroll
            for (int mt = 0; mt < MT_BLK; ++mt) {
              v[2 * mt] = o[cb * MT_BLK + mt][j][rho] * ounit;
              v[2 * mt + 1] = o[cb * MT_BLK + mt][j][rho + 2] * ounit;
            }
            const int d0 = cb * DPB + (DPB / 8) * g4;
#pragma unroll
            for (int q4 = 0; q4 < DPB / 32; ++q4) {
              const float4 f = make_float4(v[4 * q4], v[4 * q4 + 1], v[4 * q4 + 2], v[4 * q4 + 3]);
              if (whole)
                finalize_store<D>(p, vscale, f, mrun[j][rho], lsum[j][rho], h.b, h.g, r, d0 + 4 * q4);
              else if (cluster)
                *reinterpret_cast<float4*>(cp_o + (size_t)r * D + d0 + 4 * q4) = f;
              else
                *reinterpret_cast<float4*>(p.part_o + ((size_t)slot * p.Rpad + r) * D + d0 + 4 * q4) = f;
            }
          }
          if (g4 == 0 && !whole) {
            const float2 ml = make_float2(mrun[j][rho], lsum[j][rho]);
            if (cluster)
              *reinterpret_cast<float2*>(cp_ml + 2 * r) = ml;
            else
              *reinterpret_cast<float2*>(p.part_ml + ((size_t)slot * p.Rpad + r) * 2) = ml;
          }
        }
    } else {
      // several token groups: merge through the stage buffer
      float* mb_o = reinterpret_cast<float*>(sm.base + (sm.stage(s, p) - sm.base_u32));
      float* mb_ml = reinterpret_cast<float*>(sm.base + p.off_mml);
      named_bar(1, nthr);  // every warp is done reading stage s
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int rho = 0; rho < 2; ++rho) {
          const int r = row_of(j, rho);
          if (g4 == 0) {
            mb_ml[((size_t)wt * p.Rpad + r) * 2 + 0] = mrun[j][rho];
            mb_ml[((size_t)wt * p.Rpad + r) * 2 + 1] = lsum[j][rho];
          }
#pragma unroll
          for (int cb = 0; cb < NCH; ++cb) {
            float v[DPB / 8];
#pragma unroll
            for (int mt = 0; mt < MT_BLK; ++mt) {
              v[2 * mt] = o[cb * MT_BLK + mt][j][rho] * ounit;
              v[2 * mt + 1] = o[cb * MT_BLK + mt][j][rho + 2] * ounit;
            }
            float4* dst = reinterpret_cast<float4*>(mb_o + ((size_t)wt * p.Rpad + r) * D);
            const int c0 = (cb * DPB + (DPB / 8) * g4) / 4;
#pragma unroll
            for (int q4 = 0; q4 < DPB / 32; ++q4)
              dst[(c0 + q4) ^ merge_swz(r)] = make_float4(v[4 * q4], v[4 * q4 + 1], v[4 * q4 + 2], v[4 * q4 + 3]);
          }
        }
      named_bar(1, nthr);
      const int E = p.R * (D / 4);
      // per element, the token groups' shared loads are issued before any is
      // used; at most kMaxTokenWarps token groups
      for (int e = threadIdx.x; e < E; e += nthr) {
        const int r = e / (D / 4);
        const int d = (e % (D / 4)) * 4;
        const int c = (e % (D / 4)) ^ merge_swz(r);
        float2 mlw[kMaxTokenWarps];
        float4 ow[kMaxTokenWarps];
#pragma unroll
        for (int w = 0; w < kMaxTokenWarps; ++w) {
          if (w < p.Wt) {
            mlw[w] = *reinterpret_cast<const float2*>(mb_ml + ((size_t)w * p.Rpad + r) * 2);
            ow[w] = reinterpret_cast<const float4*>(mb_o + ((size_t)w * p.Rpad + r) * D)[c];
          } else {
            mlw[w] = make_float2(-INFINITY, 0.f);
            ow[w] = make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kMaxTokenWarps; ++w) M = fmaxf(M, mlw[w].x);
        float L = 0.f;
        float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
        if (M != -INFINITY) {
#pragma unroll
          for (int w = 0; w < kMaxTokenWarps; ++w) {
            if (w < p.Wt) {
              const float a = ex2(mlw[w].x - M);
              L = fmaf(mlw[w].y, a, L);
              O.x = fmaf(ow[w].x, a, O.x);
              O.y = fmaf(ow[w].y, a, O.y);
              O.z = fmaf(ow[w].z, a, O.z);
              O.w = fmaf(ow[w].w, a, O.w);
            }
          }
        }
        if (whole) {
          finalize_store<D>(p, vscale, O, M, L, h.b, h.g, r, d);
        } else if (cluster) {
          *reinterpret_cast<float4*>(cp_o + (size_t)r * D + d) = O;
          if (d == 0) *reinterpret_cast<float2*>(cp_ml + 2 * r) = make_float2(M, L);
        } else {
          *reinterpret_cast<float4*>(p.part_o + ((size_t)slot * p.Rpad + r) * D + d) = O;
          if (d == 0) *reinterpret_cast<float2*>(p.part_ml + ((size_t)slot * p.Rpad + r) * 2) = make_float2(M, L);
        }
      }
      // the stage buffer was written through the generic proxy; order that
      // before the producer's next TMA write into it
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      named_bar(1, nthr);  // the stage buffer and the (max, sum) area are read
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.empty(s, p));
    }
    if (whole || cluster) return;
    if (p.merge == kMergeReducer) {
      if (threadIdx.x == 0 && slot == md.s0) p.unit_desc[h.unit] = make_int4(md.nseg, md.s0, md.sbase, md.sstride);
    } else if (p.merge == kMergeLastArriver) {
      // Publish the partial, count it, and merge the unit here if this was
      // its last partial. A CTA has at most two split segments: its first
      // (the end of a unit others began) and its last (the start of a unit
      // others finish), so it runs at most one merge in mid-stream.
      __threadfence();
      named_bar(1, nthr);
      if (threadIdx.x == 0) arrive(h.b, h.g, h.unit, md);
      named_bar(1, nthr);
      run_queue(nthr);
    }
  }

  __device__ void arrive(int b, int g, int unit, const MergeDesc& md) { la_arrive(p, sm, b, g, unit, md); }
  __device__ void run_queue(int nthr) { la_run_queue<D>(p, sm, vscale, nthr); }
  __device__ void cluster_merge(int unit, int tid, int nthr) { cluster_merge_unit<D>(p, sm, vscale, unit, tid, nthr); }

  __device__ void run() {
    int n = 0;
    StageView h;
    while (true) {
      const int s = n % p.NS;
      bool got = mbar_wait(sm.full(s, p), (n / p.NS) & 1);
      got = __all_sync(0xffffffffu, got);
      if (!got) {
        if (lane == 0) {
          flag_status(p, kStatusTimeout);
          sm.misc(p)[0] |= 1;
        }
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
      if (p.topk > 0) {
        const int4 h2 = lds128i(ha + 32);
        h.m0 = (unsigned)h2.x;
        h.m1 = (unsigned)h2.y;
        h.m2 = (unsigned)h2.z;
        h.m3 = (unsigned)h2.w;
      }
      int slot = 0;
      MergeDesc md{1, 0, 0, 0};
      if (h.flags & kSegLast) {
        const int4 h3 = lds128i(ha + 48);
        const int sstride = lds128i(ha + 64).x;
        slot = h3.x;
        md = MergeDesc{h3.y, h3.z, h3.w, sstride};
      }
      if ((h.flags & kSegFirst) && !begin_segment(h.L)) {
        if (lane == 0) {
          flag_status(p, kStatusTimeout);
          sm.misc(p)[0] |= 1;
        }
        break;
      }
      const uint32_t kst = sm.stage(s, p);
      const uint32_t vst = kst + (uint32_t)p.TT * ROWB * NCH;
      const uint32_t sst = kst + p.off_scale;
      const int steps = p.TT / (16 * TW);
      for (int j = wt; j < steps; j += p.Wt) step(h, kst, vst, sst, j * TW);
      if (h.flags & kSegLast) {
        end_segment(h, slot, md, s);  // hands stage s back itself
      } else {
        __syncwarp();
        if (lane == 0) mbar_arrive(sm.empty(s, p));
      }
      ++n;
    }
  }

};

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// MAXW: warps per CTA the instantiation is built for (5: up to 4 consumer
// warps, two CTAs per SM at head_dim 64/128 and FP8 head_dim 256; 9: up to 8
// row-slice warps).
template <bool FP8, int D, int NT, bool VTOK, int TW, int MAXW, bool QF16 = false, bool FP4 = false, bool TV = false>
__global__ void __launch_bounds__(MAXW * 32, (MAXW == 5 && (D <= 128 || FP8)) ? 2 : 1) pa_tile_kernel(const __grid_constant__ PaParams p,
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
  if (warp == 0) prefetch_params(p);
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.NS; ++s) {
      // sparse stages: the header arrival and one copy arrival per producer lane
      mbar_init(sm.full(s, p), p.topk > 0 ? 33 : 1);
      mbar_init(sm.empty(s, p), p.NCW);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(sm.qfull(i, p), 1);
      mbar_init(sm.qempty(i, p), p.NCW);
    }
    for (int i = 0; i < 16; ++i) sm.misc(p)[i] = 0;
    fence_barrier_init();
  }
  __syncthreads();
  constexpr int ELT = FP8 ? 1 : 2;
  constexpr int NCH = FP4 ? 1 : D * ELT / 128;
  if (warp == p.NCW) {
    Producer<ELT, NCH, FP4 ? 64 : 128> prod(p, &tmK, &tmV, sm);
    prod.run();
    if (p.merge == kMergeCluster) {
      cluster_sync_all();
      cluster_sync_all();
    }
  } else {
    Consumer<FP8, D, NT, VTOK, TW, QF16, FP4, TV> cons(p, sm);
    cons.run();
    if (p.merge == kMergeCluster) {
      cluster_sync_all();
      cons.cluster_merge(blockIdx.x / p.P, threadIdx.x, p.NCW * 32);
      cluster_sync_all();
    }
  }
}

// Standalone reducer: one CTA per split unit merges its partials in order.
template <int D>
__device__ void reduce_unit(const PaParams& p) {
  const int unit = blockIdx.x;
  __shared__ int4 desc_s;
  if (threadIdx.x == 0) desc_s = p.unit_desc[unit];
  __syncthreads();
  const int4 desc = desc_s;
  if (desc.x < 2) return;
  const MergeDesc md{desc.x, desc.y, desc.z, desc.w};
  const int b = unit / p.Hkv, g = unit % p.Hkv;
  merge_elems<D>(
      p, per_tensor_vscale(p), md.nseg, b, g, threadIdx.x, blockDim.x, 0, p.R * (D / 4),
      [&](int k, int r) {
        return __ldcg(reinterpret_cast<const float2*>(p.part_ml + ((size_t)merge_slot(md, k) * p.Rpad + r) * 2));
      },
      [&](int k, int r, int d) {
        return __ldcg(reinterpret_cast<const float4*>(p.part_o + ((size_t)merge_slot(md, k) * p.Rpad + r) * D + d));
      });
  __syncthreads();
  if (threadIdx.x == 0) p.unit_desc[unit].x = 0;
}

}  // namespace dev
}  // namespace pa
