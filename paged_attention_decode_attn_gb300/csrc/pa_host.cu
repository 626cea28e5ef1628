// Host side of the C ABI: plan sizing, argument validation, TMA descriptors
// and kernel launches. No memory allocation, no stream synchronisation.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <string>

#include "pa_decode.h"
#include "pa_internal.h"

namespace {

thread_local std::string g_err;

pa_status fail(pa_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
pa_status fail(pa_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return s;
}

pa_status cuda_fail(cudaError_t e, const char* what) {
  return fail(PA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

struct pa_plan {
  pa_plan_desc desc;
  pa_plan_info info;
  pa::PaParams base;
  const void* tile_fn = nullptr;
  const void* reduce_fn = nullptr;
  void* ws = nullptr;
  size_t ws_bytes = 0;
  size_t off_part_o = 0, off_part_ml = 0, off_counters = 0, off_desc = 0, off_status = 0;
  // Launch cache: kernel attributes set once per plan, TMA descriptors of the
  // last cache pointers. A decode takes the plan as const; this cache is the
  // only state it updates, under the plan's own lock.
  mutable std::mutex cache_mu;
  mutable bool attrs_set = false;
  mutable const void* tm_k = nullptr;
  mutable const void* tm_v = nullptr;
  mutable CUtensorMap tmK, tmV;
  mutable bool tm_valid = false;
};

namespace {

// A segment's fixed cost (query rows, token-group merge, output or partial
// write) in stages of streaming, charged by the balanced schedule as virtual
// chunks per unit: about one stage on the tile consumer; about four on the
// tensor-memory consumer (Q split into its operand, pipeline drain, epilogue
// through tensor memory).
constexpr int kSegCostChunks = 1;
constexpr int kSegCostChunksTmem = 4;
// Largest dynamic shared memory a CTA may use while two CTAs share an SM, and
// with one CTA per SM.
constexpr int kSmemTwoPerSm = 112 * 1024;
constexpr int kSmemOnePerSm = 226 * 1024;

struct KernelShape {
  int nt, rw, wr, wt, ncw, rpad, elt, rb, nch, tt, tw, bh;
  int rh;   // tensor-memory consumer: query rows per softmax warpgroup
  int nwg;  // tensor-memory consumer: softmax warpgroups (2 or 4)
  bool vtok, umma;
};

// Groups of more than 16 query rows per KV head (MTP verify, wide GQA) on
// dense decode can run the tensor-memory (tcgen05) consumer: two softmax
// warpgroups over one MMA block of up to 64 rows, a producer warp and an
// MMA-issue warp. At head_dim 256 it also takes 9-16 rows (measured 9 %
// faster than the tile consumer on the long-context D256 decode at query
// length 2; at head_dim 128 the tile consumer stays ahead up to 16 rows).
bool umma_supported(const pa_plan_desc& d, int R) {
  if (d.sparse_topk > 0 || R <= (d.head_dim == 256 ? 8 : 16)) return false;
  if (d.kv_dtype == PA_KV_MXFP4) return false;  // MXFP4: the tile consumer only
  if (d.v_layout == PA_V_TRANSPOSED) return false;  // transposed V: the tile consumer only
  // BF16 caches are read in place by BF16 MMAs, whose other operand (Q) must
  // be BF16 too: FP16 queries there take the tile consumer.
  if (d.kv_dtype == PA_KV_BF16 && d.q_dtype == PA_Q_FP16) return false;
  if (d.kv_dtype == PA_KV_FP8_E4M3) return d.head_dim == 128 || d.head_dim == 256;
  return d.head_dim == 128;
}
// AUTO takes the tensor-memory consumer wherever it covers the shape.
bool use_umma(const pa_plan_desc& d, int R) {
  if (d.consumer == PA_CONSUMER_TILE || !umma_supported(d, R)) return false;
  return true;
}
constexpr int kMtpTokens = 128;   // tokens per stage (M of S^T)
constexpr int kMtpFourGroupsMaxContext = 16384;

KernelShape kernel_shape(const pa_plan_desc& d) {
  KernelShape k;
  const int G = d.num_q_heads / d.num_kv_heads;
  const int R = G * d.query_len;
  // Each consumer warp owns 8 query rows (one MMA N tile); groups of more
  // rows take more row-slice warps (up to 8 for 64 rows).
  k.nt = 1;
  k.rw = 8 * k.nt;
  k.wr = (R + k.rw - 1) / k.rw;
  k.wt = k.wr >= 4 ? 1 : 4 / k.wr;
  k.ncw = k.wr * k.wt;
  k.rpad = k.wr * k.rw;
  const bool mx = d.kv_dtype == PA_KV_MXFP4;
  // MXFP4 runs the FP8 consumer path on 64-byte rows (head_dim 128, two
  // elements per byte, one column block).
  k.elt = (d.kv_dtype == PA_KV_FP8_E4M3 || mx) ? 1 : 2;
  k.rb = mx ? d.head_dim / 2 : d.head_dim * k.elt;
  k.nch = mx ? 1 : k.rb / 128;
  // 32 KiB of K+V per ring stage; FP8 head_dim 128 steps two 16-token tiles
  // per warp (128-token stages), every other format one tile.
  int tt = 32768 / (2 * k.rb);
  k.tt = tt < 16 ? 16 : (tt > 128 ? 128 : tt);
  k.tw = ((d.kv_dtype == PA_KV_FP8_E4M3 || mx) && d.head_dim == 128) ? 2 : 1;
  k.vtok = (d.kv_dtype == PA_KV_FP8_E4M3 && d.scale_mode == PA_SCALE_PER_TOKEN) || mx;
  k.umma = use_umma(d, R);
  k.rh = 0;
  k.nwg = 0;
  if (k.umma) {
    // warpgroup w owns rows [w*rh, (w+1)*rh); 128-token stages (M = 128).
    // More than 32 rows: four warpgroups of 16 for contexts up to 16K
    // (measured 20-30 % faster on MTP4 x GQA16 with contexts up to 9000,
    // where latency decides), else two of 32 (11 % faster at 4K-64K contexts).
    const bool four = R > 32 && d.max_context_len > 0 && d.max_context_len <= kMtpFourGroupsMaxContext;
    k.rh = (R <= 32 || four) ? 16 : 32;
    k.nwg = four ? 4 : 2;
    k.nt = 2;
    k.rw = k.rh;
    k.wr = k.nwg;
    k.wt = 4;  // the four warps of a warpgroup split each stage's tokens
    k.ncw = 8;
    k.rpad = (R + 7) / 8 * 8;
    k.tt = kMtpTokens;
  }
  k.bh = d.page_size < k.tt ? d.page_size : k.tt;
  return k;
}

// Shared-memory layout for `ns` ring stages.
pa::SmemLayout smem_layout(const pa_plan_desc& d, const KernelShape& k, int ns, bool cluster, int nq) {
  pa::SmemLayout L;
  // per-token scales (4 bytes a token row: one binary32, or MXFP4's four E8M0
  // block scales) for K then V
  const bool tok_scales = d.scale_mode == PA_SCALE_PER_TOKEN || d.scale_mode == PA_SCALE_MX_BLOCK;
  L.stage_bytes = 2 * k.tt * k.rb + (tok_scales ? 1024 : 0);
  L.off_scale = 2 * k.tt * k.rb;
  L.off_stage = 0;
  size_t off = (size_t)ns * L.stage_bytes;
  L.off_k16 = L.off_v16 = L.off_q16 = L.off_p16 = 0;
  L.off_merge = (int)off;
  L.off_cpart = (int)off;  // cluster merge: this CTA's partial (O, then max/sum)
  if (k.umma) {
    // Q operand (FP8: three e4m3 terms of [D/128 chunks][RN rows][128 B];
    // BF16: [D/64 chunks][RN rows][128 B]), then the P^T slots of
    // [128 tokens][128 B] and the 2 KiB ones operand, 1024-aligned
    const int rn = k.nwg * k.rh;
    const bool fp8 = d.kv_dtype == PA_KV_FP8_E4M3;
    L.off_q16 = (int)off;
    off += fp8 ? (size_t)3 * d.head_dim * rn : (size_t)2 * d.head_dim * rn;
    off = align_up(off, 1024);
    L.off_p16 = (int)off;
    off += (size_t)(fp8 ? 3 : 2) * k.tt * 128 + 2048;  // P^T slots (FP8: three buffers; BF16: hi, lo), ones
    // the cluster partial reuses the ring, idle once the CTA's work is done
    L.off_cpart = 0;
  } else if (cluster) {
    off += align_up((size_t)k.rpad * d.head_dim * 4 + (size_t)k.rpad * 8, 128);
  }
  L.off_hdr = (int)off;
  off += (size_t)ns * 128;
  L.off_bar = (int)off;
  off += (size_t)ns * 16 + 32;  // full/empty per stage, then full/empty per Q slot
  L.off_ubar = (int)off;  // tensor-memory consumer: its fourteen pipeline barriers
  off += k.umma ? 128 : 16;
  L.off_tslot = (int)off;  // tensor-memory address written by tcgen05.alloc
  off += 16;
  L.off_rows = (int)off;  // tensor-memory consumer: per-row state (8 x 64 words)
  off += k.umma ? (size_t)8 * 64 * 4 : 0;
  off = align_up(off, 16);
  L.off_misc = (int)off;
  off += 64;
  L.off_pend = (int)off;  // queued last-arriver merges: 8 entries of 32 bytes
  off += 8 * 32;
  L.off_mml = (int)off;  // (max, sum) of the token-group warps at a segment end
  off += k.umma ? 0 : align_up((size_t)k.wt * k.rpad * 8, 128);
  L.q_slot_bytes = k.rpad * d.head_dim * 2;  // a unit's BF16 query rows
  L.nq = nq;
  L.off_q = (int)align_up(off, 16);
  off = (size_t)L.off_q + (size_t)nq * L.q_slot_bytes;
  L.total = (int)(off + 1024);  // slack for aligning the base to 1024 bytes
  return L;
}

const void* pick_tile_kernel(const pa_plan_desc& d, const KernelShape& k) {
  if (k.umma) return pa::mtp_kernel(d.kv_dtype == PA_KV_FP8_E4M3, d.head_dim, k.vtok, k.rh, k.nwg);
  if (d.kv_dtype == PA_KV_MXFP4) return pa::tile_kernel_fp4_d128(k.ncw > 4);
  if (d.kv_dtype == PA_KV_FP8_E4M3) {
    if (d.head_dim == 128) return pa::tile_kernel_fp8_d128(k.vtok, k.ncw > 4);
    return k.ncw > 4 ? nullptr : pa::tile_kernel_fp8_d256(k.vtok);
  }
  if (d.v_layout == PA_V_TRANSPOSED) return pa::tile_kernel_bf16_tv(d.head_dim, k.ncw > 4, d.q_dtype == PA_Q_FP16);
  return pa::tile_kernel_bf16(d.head_dim, k.ncw > 4, d.q_dtype == PA_Q_FP16);
}

pa_status validate_desc(const pa_plan_desc& d) {
  if (d.batch < 0) return fail(PA_ERR_INVALID_ARG, "batch must be >= 0 (got %d)", d.batch);
  if (d.num_q_heads <= 0 || d.num_kv_heads <= 0)
    return fail(PA_ERR_INVALID_ARG, "head counts must be positive (%d, %d)", d.num_q_heads, d.num_kv_heads);
  if (d.num_q_heads % d.num_kv_heads != 0)
    return fail(PA_ERR_INVALID_ARG, "num_q_heads %d is not a multiple of num_kv_heads %d", d.num_q_heads,
                d.num_kv_heads);
  if (d.head_dim != 128 && d.head_dim != 256 && !(d.head_dim == 64 && d.kv_dtype == PA_KV_BF16))
    return fail(PA_ERR_UNSUPPORTED, "head_dim %d unsupported (128 or 256; 64 with BF16 caches)", d.head_dim);
  if (d.kv_dtype == PA_KV_MXFP4 && d.head_dim != 128)
    return fail(PA_ERR_UNSUPPORTED, "MXFP4 caches support head_dim 128 (got %d)", d.head_dim);
  if (d.query_len < 1) return fail(PA_ERR_INVALID_ARG, "query_len must be >= 1 (got %d)", d.query_len);
  const long long rows = (long long)(d.num_q_heads / d.num_kv_heads) * d.query_len;
  if (rows > pa::kMaxRows)
    return fail(PA_ERR_UNSUPPORTED, "group*query_len = %lld query rows per KV head exceeds %d", rows, pa::kMaxRows);
  if (d.head_dim == 256 && rows > 32)
    return fail(PA_ERR_UNSUPPORTED, "head_dim 256 supports at most 32 query rows per KV head (got %lld)", rows);
  if (d.page_size != 16 && d.page_size != 32 && d.page_size != 64 && d.page_size != 128 && d.page_size != 256)
    return fail(PA_ERR_UNSUPPORTED, "page_size %d unsupported (16, 32, 64, 128, 256)", d.page_size);
  if (d.max_pages_per_seq < 1 || d.num_pages < 1)
    return fail(PA_ERR_INVALID_ARG, "max_pages_per_seq and num_pages must be >= 1");
  if ((long long)d.num_pages * d.num_kv_heads * d.page_size >= (1ll << 31))
    return fail(PA_ERR_UNSUPPORTED, "cache has 2^31 or more token rows per tensor");
  if ((long long)d.max_pages_per_seq * d.page_size >= (1ll << 30))
    return fail(PA_ERR_UNSUPPORTED, "max_pages_per_seq * page_size too large");
  if (d.kv_dtype != PA_KV_FP8_E4M3 && d.kv_dtype != PA_KV_BF16 && d.kv_dtype != PA_KV_MXFP4)
    return fail(PA_ERR_INVALID_ARG, "unknown kv_dtype %d", d.kv_dtype);
  if (d.scale_mode < PA_SCALE_NONE || d.scale_mode > PA_SCALE_MX_BLOCK)
    return fail(PA_ERR_INVALID_ARG, "unknown scale_mode %d", d.scale_mode);
  if ((d.kv_dtype == PA_KV_MXFP4) != (d.scale_mode == PA_SCALE_MX_BLOCK))
    return fail(PA_ERR_INVALID_ARG, "MXFP4 caches take PA_SCALE_MX_BLOCK, and only they do");
  if (d.kv_dtype == PA_KV_MXFP4 && d.sparse_topk > 0)
    return fail(PA_ERR_UNSUPPORTED, "MXFP4 caches support dense decode only");
  if (d.v_layout != PA_V_PLAIN && d.v_layout != PA_V_TRANSPOSED)
    return fail(PA_ERR_INVALID_ARG, "unknown v_layout %d", d.v_layout);
  if (d.v_layout == PA_V_TRANSPOSED) {
    if (d.kv_dtype != PA_KV_BF16)
      return fail(PA_ERR_UNSUPPORTED, "the transposed V layout is supported for BF16 caches");
    if (d.sparse_topk > 0) return fail(PA_ERR_UNSUPPORTED, "the transposed V layout supports dense decode only");
    if ((long long)d.num_pages * d.num_kv_heads * d.page_size * (d.head_dim / 64) >= (1ll << 31))
      return fail(PA_ERR_UNSUPPORTED, "transposed V cache has 2^31 or more 128-byte rows");
  }
  if (d.q_dtype != PA_Q_BF16 && d.q_dtype != PA_Q_FP16)
    return fail(PA_ERR_INVALID_ARG, "unknown q_dtype %d", d.q_dtype);
  if (d.kv_dtype == PA_KV_BF16 && d.scale_mode != PA_SCALE_NONE)
    return fail(PA_ERR_INVALID_ARG, "BF16 caches take no K/V scales");
  if (d.sparse_topk < 0) return fail(PA_ERR_INVALID_ARG, "sparse_topk must be >= 0");
  if (d.sparse_topk > 0 && d.query_len != 1)
    return fail(PA_ERR_UNSUPPORTED, "sparse decode needs query_len 1 (got %d)", d.query_len);
  if (!(d.sm_scale >= 0.f) || std::isinf(d.sm_scale))
    return fail(PA_ERR_INVALID_ARG, "sm_scale must be finite and >= 0 (0 = 1/sqrt(head_dim))");
  if (d.max_partitions < 0 || d.max_partitions > 256)
    return fail(PA_ERR_INVALID_ARG, "max_partitions must be in [0, 256]");
  if (d.merge_mode < PA_MERGE_AUTO || d.merge_mode > PA_MERGE_REDUCER)
    return fail(PA_ERR_INVALID_ARG, "unknown merge_mode %d", d.merge_mode);
  if (d.schedule < PA_SCHED_AUTO || d.schedule > PA_SCHED_PER_UNIT)
    return fail(PA_ERR_INVALID_ARG, "unknown schedule %d", d.schedule);
  if (d.consumer < PA_CONSUMER_AUTO || d.consumer > PA_CONSUMER_TMEM)
    return fail(PA_ERR_INVALID_ARG, "consumer must be PA_CONSUMER_* (got %d)", d.consumer);
  if (d.consumer == PA_CONSUMER_TMEM &&
      !umma_supported(d, d.query_len * (d.num_kv_heads > 0 ? d.num_q_heads / d.num_kv_heads : 0)))
    return fail(PA_ERR_UNSUPPORTED,
                "the tensor-memory consumer needs dense decode, 17..64 rows per KV head (9..32 at head_dim 256), "
                "FP8 head_dim 128/256 or BF16 head_dim 128 with BF16 queries");
  if (d.sm_count_override < 0 || d.ctas_per_sm_override < 0)
    return fail(PA_ERR_INVALID_ARG, "overrides must be >= 0");
  return PA_OK;
}

// Resolve schedule, partitions and merge mechanism (pure host arithmetic).
pa_status resolve_schedule(const pa_plan_desc& d, const KernelShape& k, int sm_count, int ctas_per_sm, int& sched,
                           int& merge, int& P) {
  const int units = d.batch * d.num_kv_heads;
  sched = d.schedule;
  merge = d.merge_mode;
  P = d.max_partitions;
  if (merge == PA_MERGE_DIRECT) {
    if (sched == PA_SCHED_BALANCED) return fail(PA_ERR_INVALID_ARG, "direct output needs the per-unit schedule");
    if (P > 1) return fail(PA_ERR_INVALID_ARG, "direct output needs one partition per unit");
    sched = PA_SCHED_PER_UNIT;
    P = 1;
  }
  if (merge == PA_MERGE_CLUSTER) {
    if (sched == PA_SCHED_BALANCED) return fail(PA_ERR_INVALID_ARG, "cluster merge needs the per-unit schedule");
    sched = PA_SCHED_PER_UNIT;
  }
  // Sparse decode splits each row over P CTAs while the rows leave resident
  // CTA slots free; with more rows than slots (sparse prefill) a persistent
  // balanced grid streams them, as dense decode does.
  if (sched == PA_SCHED_AUTO)
    sched = (d.sparse_topk > 0 && (long long)units <= (long long)sm_count * ctas_per_sm) ? PA_SCHED_PER_UNIT
                                                                                         : PA_SCHED_BALANCED;
  if (sched == PA_SCHED_PER_UNIT) {
    if (P == 0) {
      // Fill the resident CTA slots once: P = slots / units, in [1, 16], and
      // no more partitions than the longest unit has chunks.
      const long long slots = (long long)sm_count * ctas_per_sm;
      long long p = units > 0 ? slots / units : 1;
      if (p < 1) p = 1;
      if (p > 16) p = 16;
      long long max_tokens = d.sparse_topk > 0 ? d.sparse_topk : d.max_context_len;
      if (max_tokens > 0) {
        const long long chunks = (max_tokens + k.tt - 1) / k.tt;
        if (p > chunks) p = chunks;
      }
      if (p < 1) p = 1;
      P = (int)p;
      if (merge == PA_MERGE_CLUSTER && P < 2) P = 2;
    }
  } else {
    P = 0;
  }
  if (merge == PA_MERGE_AUTO) {
    if (sched == PA_SCHED_BALANCED)
      merge = PA_MERGE_LAST_ARRIVER;
    else
      merge = P == 1 ? PA_MERGE_DIRECT : (P <= 8 ? PA_MERGE_CLUSTER : PA_MERGE_LAST_ARRIVER);
  }
  if (merge == PA_MERGE_CLUSTER && (P < 2 || P > 16))
    return fail(PA_ERR_UNSUPPORTED, "cluster merge needs 2..16 partitions (got %d)", P);
  if (sched == PA_SCHED_PER_UNIT && P == 1) merge = PA_MERGE_DIRECT;
  return PA_OK;
}

pa_status compute_plan(pa_plan* pl, int sm_count, int ctas_override) {
  const pa_plan_desc& d = pl->desc;
  const KernelShape k = kernel_shape(d);
  pa_plan_info& in = pl->info;
  std::memset(&in, 0, sizeof in);
  pl->tile_fn = pick_tile_kernel(d, k);
  pl->reduce_fn = pa::reduce_kernel(d.head_dim);
  if (!pl->tile_fn || !pl->reduce_fn) return fail(PA_ERR_UNSUPPORTED, "no kernel for this configuration");

  // Ring depth. Kernels light enough for two CTAs per SM (at most four
  // consumer warps and 168 registers, so three warps share an SM
  // sub-partition's register file: head_dim 64/128, and FP8 head_dim 256,
  // measured 16 % faster than one CTA per SM on the long-context D256 decode)
  // get as many stages as fit 112 KiB (at least 3); the others one CTA per SM
  // and up to 226 KiB. The Q ring has two slots (the next segment's rows load
  // while the current one streams) unless that costs the third stage; one
  // slot then.
  const bool two_per_sm =
      !k.umma && k.ncw <= 4 && (d.head_dim <= 128 || d.kv_dtype == PA_KV_FP8_E4M3);
  int ns = 0, nq = 2;
  int budget = kSmemTwoPerSm;
  for (int attempt = two_per_sm ? 0 : 1; attempt < 2 && ns < 3; ++attempt) {
    budget = attempt == 0 ? kSmemTwoPerSm : kSmemOnePerSm;
    for (nq = k.umma ? 1 : 2; nq >= 1; --nq) {
      const pa::SmemLayout l0 = smem_layout(d, k, 0, d.sparse_topk > 0 || d.merge_mode == PA_MERGE_CLUSTER, nq);
      const int stage = l0.stage_bytes + 128 + 16;
      ns = (budget - l0.total) / stage;
      if (ns > 8) ns = 8;
      if (ns >= 3) break;
    }
    if (nq < 1) nq = 1;
  }
  if (ns < 2) return fail(PA_ERR_UNSUPPORTED, "shared memory too small for two ring stages");
  // the token-group warps merge their partial states inside one stage buffer
  if (!k.umma && k.wt > 1 && (size_t)k.wt * k.rpad * d.head_dim * 4 > (size_t)2 * k.tt * k.rb)
    return fail(PA_ERR_UNSUPPORTED, "token-group merge does not fit a ring stage");

  int ctas_per_sm = ctas_override;
  if (ctas_per_sm == 0) ctas_per_sm = budget == kSmemTwoPerSm ? 2 : 1;  // refined by the occupancy query

  int sched, merge, P;
  pa_status st = resolve_schedule(d, k, sm_count, ctas_per_sm, sched, merge, P);
  if (st != PA_OK) return st;
  const bool cluster = merge == PA_MERGE_CLUSTER;
  const pa::SmemLayout L = smem_layout(d, k, ns, cluster, nq);

  const int units = d.batch * d.num_kv_heads;
  const int G = d.num_q_heads / d.num_kv_heads;
  const int R = G * d.query_len;
  long long grid = sched == PA_SCHED_BALANCED ? (long long)sm_count * ctas_per_sm : (long long)units * P;
  if (units == 0) grid = 0;
  // One partial per segment of a split unit: balanced CTAs keep two slots
  // (the unit they start with, the unit they end with); per-unit plans one
  // per partition. Units one CTA covers alone are written directly.
  size_t slots = 0;
  if (sched == PA_SCHED_BALANCED)
    slots = 2 * (size_t)grid;
  else if (P > 1 && !cluster)
    slots = (size_t)units * P;
  const int kernel_merge = merge;
  const bool counters = merge == PA_MERGE_LAST_ARRIVER && slots > 0;

  // workspace: partial O, partial (max, sum), arrival counters (one 128-byte
  // line per unit), reducer descriptors, status word
  size_t off = 0;
  pl->off_part_o = off;
  off = align_up(off + slots * k.rpad * d.head_dim * 4, 256);
  pl->off_part_ml = off;
  off = align_up(off + slots * k.rpad * 8, 256);
  pl->off_counters = off;
  if (counters) off = align_up(off + (size_t)units * pa::kCounterStride * 4, 256);
  pl->off_desc = off;
  if (merge == PA_MERGE_REDUCER) off = align_up(off + (size_t)units * 16, 256);
  pl->off_status = off;
  off += 256;

  in.merge_mode = merge;
  in.schedule = sched;
  in.num_partitions = sched == PA_SCHED_PER_UNIT ? P : 0;
  in.stage_tokens = k.tt;
  in.num_stages = ns;
  in.rows = R;
  in.rows_per_warp = k.rw;
  in.row_warps = k.wr;
  in.token_warps = k.wt;
  // tensor memory: softmax warpgroups, the producer warp and the MMA warp
  in.block_threads = k.umma ? 32 * (4 * k.nwg + 2) : (k.ncw + 1) * 32;
  in.grid = (int)grid;
  in.cluster = cluster ? P : 1;
  in.ctas_per_sm = ctas_per_sm;
  in.sm_count = sm_count;
  in.launches_per_call = merge == PA_MERGE_REDUCER ? 2 : 1;
  in.units = units;
  in.consumer = k.umma ? PA_CONSUMER_TMEM : PA_CONSUMER_TILE;
  in.smem_bytes = (size_t)L.total;
  in.workspace_bytes = off;
  in.partial_slots = slots;
  in.status_offset = pl->off_status;

  pa::PaParams& p = pl->base;
  std::memset(&p, 0, sizeof p);
  p.B = d.batch;
  p.Hq = d.num_q_heads;
  p.Hkv = d.num_kv_heads;
  p.G = G;
  p.QL = d.query_len;
  p.D = d.head_dim;
  p.S = d.page_size;
  p.maxp = d.max_pages_per_seq;
  p.num_pages = d.num_pages;
  p.R = R;
  p.Rpad = k.rpad;
  p.causal = d.causal ? 1 : 0;
  p.topk = d.sparse_topk;
  p.has_sinks = d.has_sinks ? 1 : 0;
  // MXFP4 block scales travel like per-token scales (four bytes a token row)
  p.scale_mode = d.kv_dtype == PA_KV_FP8_E4M3 ? d.scale_mode
                 : d.kv_dtype == PA_KV_MXFP4 ? pa::kScalePerToken
                                             : pa::kScaleNone;
  p.q_f16 = d.q_dtype == PA_Q_FP16;
  p.v_tr = d.v_layout == PA_V_TRANSPOSED;
  const float sm_scale = d.sm_scale > 0.f ? d.sm_scale : 1.0f / std::sqrt((float)d.head_dim);
  p.sm_scale_log2 = sm_scale * 1.4426950408889634f;
  p.sched = sched;
  p.merge = kernel_merge;
  p.C = sched == PA_SCHED_BALANCED ? (int)grid : 0;
  p.seg_cost = sched == PA_SCHED_BALANCED ? (k.umma ? kSegCostChunksTmem : kSegCostChunks) : 0;
  p.P = sched == PA_SCHED_PER_UNIT ? P : 0;
  p.TT = k.tt;
  p.NS = ns;
  p.Wr = k.wr;
  p.Wt = k.wt;
  p.NCW = k.ncw;
  p.BH = k.bh;
  p.off_stage = L.off_stage;
  p.stage_bytes = L.stage_bytes;
  p.off_scale = L.off_scale;
  p.off_hdr = L.off_hdr;
  p.off_bar = L.off_bar;
  p.off_merge = L.off_merge;
  p.off_cpart = L.off_cpart;
  p.off_misc = L.off_misc;
  p.off_pend = L.off_pend;
  p.off_mml = L.off_mml;
  p.off_q = L.off_q;
  p.off_k16 = L.off_k16;
  p.off_v16 = L.off_v16;
  p.off_q16 = L.off_q16;
  p.off_p16 = L.off_p16;
  p.off_ubar = L.off_ubar;
  p.off_tslot = L.off_tslot;
  p.off_rows = L.off_rows;
  p.q_slot_bytes = L.q_slot_bytes;
  p.NQ = L.nq;
  return PA_OK;
}

// Kernel attributes (dynamic shared memory, non-portable cluster size) are
// set once per plan, on the plan's device. Caller holds pl->cache_mu.
pa_status set_kernel_attrs(const pa_plan* pl) {
  if (pl->attrs_set) return PA_OK;
  pa::DeviceGuard guard(pl->desc.device);
  cudaError_t e = guard.error();
  if (e != cudaSuccess) return cuda_fail(e, "cudaSetDevice");
  e = cudaFuncSetAttribute(pl->tile_fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl->info.smem_bytes);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(max dynamic smem)");
  if (pl->info.cluster > 8) {
    e = cudaFuncSetAttribute(pl->tile_fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(non-portable cluster)");
  }
  pl->attrs_set = true;
  return PA_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// 2-D view of a paged cache: rows = (page, kv head, slot), columns = head dims.
// A transposed V cache ([page, kv head, slot / 8, dim, slot % 8], BF16) is
// viewed as 128-byte rows of 8 dims x 8 tokens; a page is BH * D / 64 rows.
pa_status encode_cache_map(const pa_plan* pl, const void* base, CUtensorMap* tm, bool v) {
  const pa_plan_desc& d = pl->desc;
  auto fn = encode_fn();
  if (!fn) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  if (v && d.v_layout == PA_V_TRANSPOSED) {
    cuuint64_t dims[2] = {64, (cuuint64_t)d.num_pages * d.num_kv_heads * d.page_size * (d.head_dim / 64)};
    cuuint64_t strides[1] = {128};
    cuuint32_t box[2] = {64, (cuuint32_t)(pl->base.BH * (d.head_dim / 64))};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return PA_OK;
  }
  const bool mx = d.kv_dtype == PA_KV_MXFP4;
  const int elt = d.kv_dtype == PA_KV_FP8_E4M3 || mx ? 1 : 2;
  // MXFP4: rows of head_dim / 2 bytes (64), one box per page, 64-byte swizzle
  const cuuint64_t row_elems = mx ? (cuuint64_t)d.head_dim / 2 : (cuuint64_t)d.head_dim;
  cuuint64_t dims[2] = {row_elems, (cuuint64_t)d.num_pages * d.num_kv_heads * d.page_size};
  cuuint64_t strides[1] = {row_elems * elt};
  cuuint32_t box[2] = {mx ? (cuuint32_t)row_elems : (cuuint32_t)(128 / elt), (cuuint32_t)pl->base.BH};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(tm, elt == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                  const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  mx ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return PA_OK;
}

// Validate the call and launch the plan's kernel(s) on workspace `ws`.
pa_status launch(const pa_plan* pl, void* ws_ptr, void* out, const void* q, const void* k_cache, const void* v_cache,
                 const int32_t* block_table, const int32_t* ctx_lens, const int32_t* topk_idx, const float* k_scale,
                 const float* v_scale, int window, const float* sinks, void* stream) {
  const pa_plan_desc& d = pl->desc;
  if (d.batch == 0) return PA_OK;
  if (!out || !q || !k_cache || !v_cache || !block_table || !ctx_lens)
    return fail(PA_ERR_INVALID_ARG, "null tensor pointer");
  const void* ptrs[] = {out, q, k_cache, v_cache, block_table, ctx_lens, topk_idx, k_scale, v_scale, sinks};
  for (const void* ptr : ptrs)
    if (ptr && !aligned16(ptr)) return fail(PA_ERR_INVALID_ARG, "tensor pointer %p is not 16-byte aligned", ptr);
  if (d.kv_dtype == PA_KV_FP8_E4M3 && d.scale_mode != PA_SCALE_NONE && (!k_scale || !v_scale))
    return fail(PA_ERR_INVALID_ARG, "FP8 scales are required by the plan's scale_mode");
  if (d.kv_dtype == PA_KV_MXFP4 && (!k_scale || !v_scale))
    return fail(PA_ERR_INVALID_ARG, "MXFP4 caches need their block-scale arrays (k_scale, v_scale)");
  if (d.has_sinks && !sinks) return fail(PA_ERR_INVALID_ARG, "the plan has sinks but sinks is null");
  if (window < 0) return fail(PA_ERR_INVALID_ARG, "window must be >= 0");
  if (window > 0 && !d.causal && d.query_len > 1)
    return fail(PA_ERR_UNSUPPORTED, "a window with non-causal multi-token queries is not defined");
  if (!ws_ptr) return fail(PA_ERR_WORKSPACE, "no workspace bound to the plan");
  CUtensorMap tmK, tmV;
  {
    std::lock_guard<std::mutex> lock(pl->cache_mu);
    pa_status st = set_kernel_attrs(pl);
    if (st != PA_OK) return st;
    if (!pl->tm_valid || pl->tm_k != k_cache || pl->tm_v != v_cache) {
      pl->tm_valid = false;
      st = encode_cache_map(pl, k_cache, &pl->tmK, false);
      if (st != PA_OK) return st;
      st = encode_cache_map(pl, v_cache, &pl->tmV, true);
      if (st != PA_OK) return st;
      pl->tm_k = k_cache;
      pl->tm_v = v_cache;
      pl->tm_valid = true;
    }
    tmK = pl->tmK;
    tmV = pl->tmV;
  }
  pa::PaParams p = pl->base;
  uint8_t* ws = static_cast<uint8_t*>(ws_ptr);
  p.out = static_cast<uint16_t*>(out);
  p.q = static_cast<const uint16_t*>(q);
  p.block_table = block_table;
  p.ctx_lens = ctx_lens;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.sinks = d.has_sinks ? sinks : nullptr;
  p.topk_idx = topk_idx;
  p.k_cache = static_cast<const uint8_t*>(k_cache);
  p.v_cache = static_cast<const uint8_t*>(v_cache);
  p.window = d.sparse_topk > 0 ? 0 : window;
  p.part_o = reinterpret_cast<float*>(ws + pl->off_part_o);
  p.part_ml = reinterpret_cast<float*>(ws + pl->off_part_ml);
  p.counters = reinterpret_cast<int*>(ws + pl->off_counters);
  p.unit_desc = reinterpret_cast<int4*>(ws + pl->off_desc);
  p.status = reinterpret_cast<int*>(ws + pl->off_status);

  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3((unsigned)pl->info.grid, 1, 1);
  cfg.blockDim = dim3((unsigned)pl->info.block_threads, 1, 1);
  cfg.dynamicSmemBytes = pl->info.smem_bytes;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  if (pl->info.cluster > 1) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)pl->info.cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  void* args[] = {&p, &tmK, &tmV};
  cudaError_t e = cudaLaunchKernelExC(&cfg, pl->tile_fn, args);
  if (e != cudaSuccess) return cuda_fail(e, "tile kernel launch");
  if (pl->info.merge_mode == PA_MERGE_REDUCER) {
    cudaLaunchConfig_t rc;
    std::memset(&rc, 0, sizeof rc);
    rc.gridDim = dim3((unsigned)pl->info.units, 1, 1);
    rc.blockDim = dim3(128, 1, 1);
    rc.stream = static_cast<cudaStream_t>(stream);
    void* rargs[] = {&p};
    e = cudaLaunchKernelExC(&rc, pl->reduce_fn, rargs);
    if (e != cudaSuccess) return cuda_fail(e, "reducer launch");
  }
  return PA_OK;
}

}  // namespace

namespace pa {

// Decode with an explicit workspace in place of the plan's bound one. The
// plan's launch cache (kernel attributes, tensor maps) is shared with
// pa_decode; its bound workspace is neither used nor changed.
pa_status launch_on_workspace(const pa_plan* plan, void* ws, size_t ws_bytes, void* out, const void* q,
                              const void* k_cache, const void* v_cache, const int32_t* block_table,
                              const int32_t* ctx_lens, const float* k_scale, const float* v_scale, int window,
                              const float* sinks, void* stream) {
  if (ws_bytes < plan->info.workspace_bytes) return fail(PA_ERR_WORKSPACE, "scratch smaller than the plan's workspace");
  return launch(plan, ws, out, q, k_cache, v_cache, block_table, ctx_lens, nullptr, k_scale, v_scale, window, sinks,
                stream);
}

// Record a failure message for pa_last_error() and return the status.
pa_status set_error(pa_status status, const char* message) { return fail(status, "%s", message); }

// Workspace bytes of a plan, the offset from which its workspace must start
// zero-filled (arrival counters, reducer descriptors, status word), and its device.
size_t plan_workspace_layout(const pa_plan* plan, size_t* zero_from, int* device, int* sparse) {
  *zero_from = plan->off_counters;
  *device = plan->desc.device;
  *sparse = plan->desc.sparse_topk > 0;
  return plan->info.workspace_bytes;
}

}  // namespace pa

extern "C" {

pa_status pa_plan_create(const pa_plan_desc* desc, pa_plan_t** out) {
  if (!desc || !out) return fail(PA_ERR_INVALID_ARG, "null argument");
  *out = nullptr;
  pa_status st = validate_desc(*desc);
  if (st != PA_OK) return st;
  pa_plan* pl = new (std::nothrow) pa_plan();
  if (!pl) return fail(PA_ERR_INVALID_ARG, "out of host memory");
  pl->desc = *desc;
  int sm_count = desc->sm_count_override;
  const bool host_only = desc->sm_count_override > 0 && desc->ctas_per_sm_override > 0;
  if (sm_count == 0) {
    cudaError_t e = cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, desc->device);
    if (e != cudaSuccess) {
      delete pl;
      return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
    }
  }
  st = compute_plan(pl, sm_count, desc->ctas_per_sm_override);
  if (st == PA_OK && !host_only && desc->ctas_per_sm_override == 0 && pl->info.schedule == PA_SCHED_BALANCED) {
    // Size the persistent grid by the measured occupancy of the chosen kernel.
    st = set_kernel_attrs(pl);
    int n = 0;
    if (st == PA_OK) {
      pa::DeviceGuard guard(desc->device);
      cudaError_t e = guard.error();
      if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, pl->tile_fn, pl->info.block_threads,
                                                         pl->info.smem_bytes);
      if (e != cudaSuccess) st = cuda_fail(e, "occupancy query");
    }
    if (st == PA_OK) {
      if (n < 1) n = 1;
      if (n != pl->info.ctas_per_sm) {
        const bool attrs = pl->attrs_set;
        st = compute_plan(pl, sm_count, n);
        pl->attrs_set = attrs;
      }
    }
  }
  if (st != PA_OK) {
    delete pl;
    return st;
  }
  *out = pl;
  return PA_OK;
}

size_t pa_plan_workspace_bytes(const pa_plan_t* plan) { return plan ? plan->info.workspace_bytes : 0; }

pa_status pa_plan_set_workspace(pa_plan_t* plan, void* dev_ptr, size_t bytes) {
  if (!plan) return fail(PA_ERR_INVALID_ARG, "null plan");
  if (!dev_ptr) return fail(PA_ERR_WORKSPACE, "null workspace");
  if ((reinterpret_cast<uintptr_t>(dev_ptr) & 255u) != 0)
    return fail(PA_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  if (bytes < plan->info.workspace_bytes)
    return fail(PA_ERR_WORKSPACE, "workspace has %zu bytes, the plan needs %zu", bytes, plan->info.workspace_bytes);
  plan->ws = dev_ptr;
  plan->ws_bytes = bytes;
  return PA_OK;
}

pa_status pa_plan_get_info(const pa_plan_t* plan, pa_plan_info* info) {
  if (!plan || !info) return fail(PA_ERR_INVALID_ARG, "null argument");
  *info = plan->info;
  return PA_OK;
}

void pa_plan_destroy(pa_plan_t* plan) { delete plan; }

pa_status pa_decode(void* out, const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                    const int32_t* ctx_lens, const float* k_scale, const float* v_scale, int window,
                    const float* sinks, const pa_plan_t* plan, void* stream) {
  if (!plan) return fail(PA_ERR_INVALID_ARG, "null plan");
  if (plan->desc.sparse_topk > 0) return fail(PA_ERR_INVALID_ARG, "the plan is for sparse decode");
  return launch(plan, plan->ws, out, q, k_cache, v_cache, block_table, ctx_lens, nullptr, k_scale, v_scale, window,
                sinks, stream);
}

pa_status pa_decode_sparse(void* out, const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* block_table, const int32_t* ctx_lens, const int32_t* topk_idx,
                           const float* k_scale, const float* v_scale, const float* sinks, const pa_plan_t* plan,
                           void* stream) {
  if (!plan) return fail(PA_ERR_INVALID_ARG, "null plan");
  if (plan->desc.sparse_topk == 0) return fail(PA_ERR_INVALID_ARG, "the plan is for dense decode");
  if (!topk_idx) return fail(PA_ERR_INVALID_ARG, "null topk_idx");
  return launch(plan, plan->ws, out, q, k_cache, v_cache, block_table, ctx_lens, topk_idx, k_scale, v_scale, 0, sinks,
                stream);
}

const char* pa_strerror(pa_status s) {
  switch (s) {
    case PA_OK: return "success";
    case PA_ERR_INVALID_ARG: return "invalid argument";
    case PA_ERR_UNSUPPORTED: return "unsupported configuration";
    case PA_ERR_WORKSPACE: return "workspace missing or too small";
    case PA_ERR_CUDA: return "CUDA error";
    case PA_ERR_DEVICE_STATUS: return "kernel reported an error in its status word";
  }
  return "unknown status";
}

const char* pa_last_error(void) { return g_err.c_str(); }

}  // extern "C"
