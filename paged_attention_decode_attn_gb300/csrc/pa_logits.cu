// Indexer logits for sm_103a: FP8 queries against an FP8 KV list, a ReLU x
// weight epilogue reduced over the heads (PR "[FlyDSL] fp8_mqa_logits gfx942:
// add LDS-staged variant, use it by default": Summary and Changes).
//
// One CTA takes a block of RB query rows (RB x H = 256 MMA columns) and a
// share of the 128-token KV tiles their windows cover:
//  * warp 0 loads the block's query rows once (TMA, 128-byte swizzle) and
//    streams KV tiles through a shared-memory ring;
//  * warp 1 issues S^T = K . Q^T per tile as tcgen05 kind::f8f6f4 MMAs (M = 128
//    tokens, N = 256 (row, head) columns, K = 128 dims in four steps) into one
//    of two tensor-memory buffers;
//  * the epilogue warps (16; 8 at 128 heads) read S^T back, four (two) per
//    tensor-memory lane quarter, each a 64-column (128-column) slice of whole
//    rows, form sum_h w[r][h] * max(0, s) per (row, token), apply the token's
//    scale and the row's window, and store the logits rows (32 consecutive
//    tokens per warp store).
// Every wait is bounded; a wait that runs out sets a bit in the status word
// and the roles unwind.
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cstring>
#include <mutex>

#include "pa_decode.h"
#include "pa_internal.h"
#include "pa_tc.cuh"

namespace pa {
namespace dev {

// epilogue warps per CTA, and the (row, head) columns each one reduces
__host__ __device__ constexpr int lg_epi_warps(int H) { return H == 128 ? 8 : 16; }
__host__ __device__ constexpr int lg_threads(int H) { return 32 * (2 + lg_epi_warps(H)); }
constexpr int kLgTile = 128;     // KV tokens per tile (M of S^T)
constexpr int kLgStages = 6;     // KV ring depth
constexpr int kLgN = 256;        // (row, head) columns per row block
constexpr int kLgStatusTimeout = 1;

// Shared memory, from a 1024-byte-aligned base: the block's query rows
// (256 x 128 e4m3 bytes), the KV ring, the block's head weights, barriers and
// the tensor-memory address slot.
constexpr uint32_t kLgOffQ = 0;
constexpr uint32_t kLgOffK = kLgN * 128;
constexpr uint32_t kLgStageBytes = kLgTile * 128;
constexpr uint32_t kLgOffW = kLgOffK + kLgStages * kLgStageBytes;
constexpr uint32_t kLgOffBar = kLgOffW + kLgN * 4;
constexpr uint32_t kLgBars = 2 * kLgStages + 6;
constexpr uint32_t kLgOffSlot = kLgOffBar + kLgBars * 8;
constexpr uint32_t kLgSmemBytes = kLgOffSlot + 16 + 1024;  // + slack to align the base

struct LogitsParams {
  float* logits;
  const float* kv_scale;
  const float* weights;
  const int* ks;
  const int* ke;
  int* status;
  int rows, n_kv, stride, clean;
};

__device__ __forceinline__ void tma_load_2d_l(uint32_t dst, const CUtensorMap* tm, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ uint64_t desc_add(uint64_t d, uint32_t bytes) { return d + (uint64_t)(bytes >> 4); }
__device__ __forceinline__ void lg_tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
}
// Two FP32 lanes in one 64-bit register, and their packed FMA (fma.rn.f32x2):
// one instruction for two products.
__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ float f32x2_sum(uint64_t a) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(a));
  return lo + hi;
}
// acc += sum over n of w[n] * max(0, s[n]) (s: tensor-memory words), even
// and odd n in the two lanes of acc
template <int NV>
__device__ __forceinline__ uint64_t lg_relu_dot(const uint32_t (&v)[NV], const float* w, uint64_t acc) {
#pragma unroll
  for (int x = 0; x < NV; x += 4) {
    const float4 w4 = *reinterpret_cast<const float4*>(w + x);
    acc = fma_f32x2(f32x2(w4.x, w4.y),
                    f32x2(fmaxf(__uint_as_float(v[x]), 0.f), fmaxf(__uint_as_float(v[x + 1]), 0.f)), acc);
    acc = fma_f32x2(f32x2(w4.z, w4.w),
                    f32x2(fmaxf(__uint_as_float(v[x + 2]), 0.f), fmaxf(__uint_as_float(v[x + 3]), 0.f)), acc);
  }
  return acc;
}

struct LgBars {
  uint32_t base;
  __device__ __forceinline__ uint32_t full(int s) const { return base + 8u * (uint32_t)s; }
  __device__ __forceinline__ uint32_t empty(int s) const { return base + 8u * (uint32_t)(kLgStages + s); }
  __device__ __forceinline__ uint32_t sfull(int b) const { return base + 8u * (uint32_t)(2 * kLgStages + b); }
  __device__ __forceinline__ uint32_t sfree(int b) const { return base + 8u * (uint32_t)(2 * kLgStages + 2 + b); }
  __device__ __forceinline__ uint32_t qfull() const { return base + 8u * (uint32_t)(2 * kLgStages + 4); }
  __device__ __forceinline__ uint32_t drained() const { return base + 8u * (uint32_t)(2 * kLgStages + 5); }
};

__device__ __forceinline__ void lg_fail(const LogitsParams& p, volatile int* flag) {
  *flag = 1;
  if (p.status) atomicOr(p.status, kLgStatusTimeout);
}

// -inf over columns [c0, c1) of the block's rows (the parts of [0, num_kv)
// that no tile of this block covers), by `nthr` threads starting at `tid`.
__device__ __forceinline__ void lg_fill(const LogitsParams& p, int RB, int r0, int c0, int c1, int tid, int nthr) {
  if (c1 <= c0) return;
  const float ninf = -INFINITY;
  for (int rl = 0; rl < RB; ++rl) {
    const int r = r0 + rl;
    if (r >= p.rows) break;
    float* row = p.logits + (size_t)r * p.stride;
    // c0 is a multiple of 128; quads up to the last whole one, then singles
    const int q1 = c0 + ((c1 - c0) & ~3);
    for (int c = c0 + 4 * tid; c < q1; c += 4 * nthr)
      *reinterpret_cast<float4*>(row + c) = make_float4(ninf, ninf, ninf, ninf);
    for (int c = q1 + tid; c < c1; c += nthr) row[c] = ninf;
  }
}

template <int H>
__global__ void __launch_bounds__(lg_threads(H), 1)
    pa_logits_kernel(const __grid_constant__ LogitsParams p, const __grid_constant__ CUtensorMap tmQ,
                     const __grid_constant__ CUtensorMap tmK) {
  constexpr int RB = kLgN / H;                // query rows per block
  constexpr int NE = lg_epi_warps(H);         // epilogue warps
  constexpr int NT = lg_threads(H);           // threads per CTA
  constexpr int RPW = RB / (NE / 4);          // rows per epilogue warp (whole rows)
  static_assert(RPW >= 1 && RPW * (NE / 4) == RB, "epilogue slices hold whole rows");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sbase = smem_raw + (base - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = blockIdx.x * RB;
  // the block's tile range: the union of its rows' windows, clipped to [0, num_kv)
  int lo = INT_MAX, hi = 0;
  for (int rl = 0; rl < RB; ++rl) {
    const int r = r0 + rl;
    if (r >= p.rows) break;
    const int a = max(0, __ldg(p.ks + r)), e = min(p.n_kv, __ldg(p.ke + r));
    if (e > a) {
      lo = min(lo, a);
      hi = max(hi, e);
    }
  }
  int t_lo = 0, t_hi = 0;
  if (hi > 0 && lo < hi) {
    t_lo = lo / kLgTile;
    t_hi = (hi + kLgTile - 1) / kLgTile;
  }
  const int n = t_hi - t_lo;
  const int chunk = (n + (int)gridDim.y - 1) / (int)gridDim.y;
  const int k0 = t_lo + min(n, (int)blockIdx.y * chunk), k1 = t_lo + min(n, (int)(blockIdx.y + 1) * chunk);
  const int nt = k1 - k0;
  // uncovered columns of the block's rows: -inf, by the first split
  if (p.clean && blockIdx.y == 0) {
    lg_fill(p, RB, r0, 0, min(p.n_kv, t_lo * kLgTile), threadIdx.x, NT);
    lg_fill(p, RB, r0, min(p.n_kv, t_hi * kLgTile), p.n_kv, threadIdx.x, NT);
  }
  if (nt <= 0) return;  // uniform across the CTA: nothing waits on this CTA

  LgBars bars{base + kLgOffBar};
  volatile int* fail_flag = reinterpret_cast<volatile int*>(sbase + kLgOffSlot + 8);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kLgStages; ++s) {
      mbar_init(bars.full(s), 1);
      mbar_init(bars.empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bars.sfull(b), 1);
      mbar_init(bars.sfree(b), NE);
    }
    mbar_init(bars.qfull(), 1);
    mbar_init(bars.drained(), 1);
    *fail_flag = 0;
    fence_barrier_init();
  }
  // head weights of the block's rows (rows past the end: 0)
  float* wsm = reinterpret_cast<float*>(sbase + kLgOffW);
  for (int i = threadIdx.x; i < kLgN; i += NT) {
    const int r = r0 + i / H;
    wsm[i] = r < p.rows ? __ldg(p.weights + (size_t)r * H + i % H) : 0.f;
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(base + kLgOffSlot),
                 "r"(2 * kLgN)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sbase + kLgOffSlot);

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmQ)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmK)) : "memory");
      mbar_arrive_tx(bars.qfull(), (uint32_t)kLgN * 128u);
      tma_load_2d_l(base + kLgOffQ, &tmQ, 0, r0 * H, bars.qfull());
      for (int k = 0; k < nt; ++k) {
        const int s = k % kLgStages;
        if (!mbar_wait(bars.empty(s), ((k / kLgStages) & 1) ^ 1) || *fail_flag) {
          lg_fail(p, fail_flag);
          break;
        }
        mbar_arrive_tx(bars.full(s), kLgStageBytes);
        tma_load_2d_l(base + kLgOffK + (uint32_t)s * kLgStageBytes, &tmK, 0, (k0 + k) * kLgTile, bars.full(s));
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issue
    if (lane == 0) {
      constexpr uint32_t idesc = umma_idesc_ab(false, kLgTile, kLgN, false, false);  // e4m3 x e4m3, K-major
      const uint64_t dq = umma_sdesc(base + kLgOffQ, 16, 1024);
      bool good = mbar_wait(bars.qfull(), 0);
      for (int k = 0; k < nt && good; ++k) {
        const int s = k % kLgStages, b = k & 1;
        good = mbar_wait(bars.full(s), (k / kLgStages) & 1);
        if (good && k >= 2) good = mbar_wait(bars.sfree(b), ((k - 2) >> 1) & 1);
        if (!good || *fail_flag) break;
        tc_fence_after();
        const uint64_t dk = umma_sdesc(base + kLgOffK + (uint32_t)s * kLgStageBytes, 16, 1024);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          umma_f8(tmem + (uint32_t)(b * kLgN), desc_add(dk, 32u * j), desc_add(dq, 32u * j), idesc, j > 0 ? 1u : 0u);
        umma_commit(bars.empty(s));
        umma_commit(bars.sfull(b));
      }
      if (!good) lg_fail(p, fail_flag);
      // every issued MMA completes before the CTA frees tensor memory
      umma_commit(bars.drained());
      if (!mbar_wait_spin(bars.drained(), 0)) lg_fail(p, fail_flag);
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int e = warp - 2;
    const int quarter = warp & 3;  // the tensor-memory lanes this warp may read
    const int half = e >> 2;       // which slice of the block's rows
    const int tok = 32 * quarter + lane;
    const uint32_t lane_addr = (uint32_t)(32 * quarter) << 16;
    int wks[RPW], wke[RPW];
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
      const int r = r0 + half * RPW + i;
      const bool ok = r < p.rows;
      wks[i] = ok ? __ldg(p.ks + r) : 0;
      wke[i] = ok ? __ldg(p.ke + r) : 0;
    }
    float sc_next = 0.f;
    {
      const int j = k0 * kLgTile + tok;
      sc_next = j < p.n_kv ? __ldg(p.kv_scale + j) : 0.f;
    }
    for (int k = 0; k < nt; ++k) {
      const int b = k & 1;
      const int j = (k0 + k) * kLgTile + tok;
      const float sc = sc_next;
      if (k + 1 < nt) {
        const int jn = j + kLgTile;
        sc_next = jn < p.n_kv ? __ldg(p.kv_scale + jn) : 0.f;
      }
      bool got = mbar_wait(bars.sfull(b), (k >> 1) & 1);
      got = __all_sync(0xffffffffu, got);
      if (!got || *fail_flag) {
        if (lane == 0) lg_fail(p, fail_flag);
        break;
      }
      tc_fence_after();
      float acc[RPW];
#pragma unroll
      for (int i = 0; i < RPW; ++i) {
        uint64_t a2 = f32x2(0.f, 0.f);
        const int col0 = b * kLgN + (half * RPW + i) * H;
        const float* w = wsm + (half * RPW + i) * H;
        if constexpr (H == 16) {
          uint32_t v[16];
          lg_tmem_ld16(tmem + lane_addr + (uint32_t)col0, v);
          tmem_wait_ld();
          a2 = lg_relu_dot<16>(v, w, a2);
        } else {
          // 64 columns (two loads) per wait
#pragma unroll
          for (int h0 = 0; h0 < H; h0 += 64) {
            uint32_t va[32], vb[32];
            tmem_ld32(tmem + lane_addr + (uint32_t)(col0 + h0), va);
            if (h0 + 32 < H) tmem_ld32(tmem + lane_addr + (uint32_t)(col0 + h0 + 32), vb);
            tmem_wait_ld();
            a2 = lg_relu_dot<32>(va, w + h0, a2);
            if (h0 + 32 < H) a2 = lg_relu_dot<32>(vb, w + h0 + 32, a2);
          }
        }
        acc[i] = f32x2_sum(a2);
      }
      // S buffer b is read: the MMA of tile k + 2 may overwrite it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.sfree(b));
      if (j < p.n_kv) {
#pragma unroll
        for (int i = 0; i < RPW; ++i) {
          const int r = r0 + half * RPW + i;
          if (r >= p.rows) break;
          float* dst = p.logits + (size_t)r * p.stride + j;
          if (j >= wks[i] && j < wke[i])
            *dst = acc[i] * sc;
          else if (p.clean)
            *dst = -INFINITY;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(2 * kLgN) : "memory");
  }
}

}  // namespace dev

namespace {

PFN_cuTensorMapEncodeTiled_v12000 logits_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// 2-D byte view [rows, 128] with 128-byte swizzled boxes of box_rows rows.
bool encode_rows(CUtensorMap* tm, const void* base, long long rows, int box_rows) {
  auto fn = logits_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {128, (cuuint64_t)rows};
  cuuint64_t strides[1] = {128};
  cuuint32_t box[2] = {128, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16p(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int kMaxLogitsDevices = 64;
std::mutex g_logits_attr_mutex;
bool g_logits_attr_set[kMaxLogitsDevices];

}  // namespace
}  // namespace pa

extern "C" pa_status pa_mqa_logits(float* logits, int logits_stride, const void* q, const void* kv,
                                   const float* kv_scale, const float* weights, const int32_t* ks,
                                   const int32_t* ke, int rows, int num_heads, int head_dim, int num_kv,
                                   int clean_logits, int32_t* status, int device, void* stream) {
  using namespace pa;
  if (rows < 0 || num_kv < 0) return set_error(PA_ERR_INVALID_ARG, "rows and num_kv must be >= 0");
  if (num_heads != 16 && num_heads != 32 && num_heads != 64 && num_heads != 128)
    return set_error(PA_ERR_UNSUPPORTED, "num_heads must be 16, 32, 64 or 128");
  if (head_dim != 128) return set_error(PA_ERR_UNSUPPORTED, "head_dim must be 128");
  if (logits_stride < num_kv || logits_stride % 4 != 0)
    return set_error(PA_ERR_INVALID_ARG, "logits_stride must be >= num_kv and a multiple of 4");
  if (device < 0 || device >= kMaxLogitsDevices) return set_error(PA_ERR_INVALID_ARG, "device ordinal out of range");
  if (rows == 0 || num_kv == 0) return PA_OK;
  const void* ptrs[] = {logits, q, kv, kv_scale, weights, ks, ke};
  for (const void* ptr : ptrs)
    if (!ptr || !aligned16p(ptr)) return set_error(PA_ERR_INVALID_ARG, "null or misaligned (16-byte) pointer");
  if (status && (reinterpret_cast<uintptr_t>(status) & 3u)) return set_error(PA_ERR_INVALID_ARG, "misaligned status");
  if ((long long)rows * num_heads >= (1ll << 31)) return set_error(PA_ERR_INVALID_ARG, "rows * num_heads too large");

  DeviceGuard guard(device);
  cudaError_t e = guard.error();
  if (e != cudaSuccess) return set_error(PA_ERR_CUDA, cudaGetErrorString(e));
  {
    std::lock_guard<std::mutex> lock(g_logits_attr_mutex);
    if (!g_logits_attr_set[device]) {
      const void* fns[] = {reinterpret_cast<const void*>(&dev::pa_logits_kernel<16>),
                           reinterpret_cast<const void*>(&dev::pa_logits_kernel<32>),
                           reinterpret_cast<const void*>(&dev::pa_logits_kernel<64>),
                           reinterpret_cast<const void*>(&dev::pa_logits_kernel<128>)};
      for (const void* f : fns) {
        e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dev::kLgSmemBytes);
        if (e != cudaSuccess) return set_error(PA_ERR_CUDA, cudaGetErrorString(e));
      }
      g_logits_attr_set[device] = true;
    }
  }
  CUtensorMap tmQ, tmK;
  if (!encode_rows(&tmQ, q, (long long)rows * num_heads, dev::kLgN) || !encode_rows(&tmK, kv, num_kv, dev::kLgTile))
    return set_error(PA_ERR_CUDA, "cuTensorMapEncodeTiled failed");
  dev::LogitsParams p;
  std::memset(&p, 0, sizeof p);
  p.logits = logits;
  p.kv_scale = kv_scale;
  p.weights = weights;
  p.ks = ks;
  p.ke = ke;
  p.status = status;
  p.rows = rows;
  p.n_kv = num_kv;
  p.stride = logits_stride;
  p.clean = clean_logits != 0;
  const int RB = dev::kLgN / num_heads;
  const int nblk = (rows + RB - 1) / RB;
  const void* fn = num_heads == 16   ? reinterpret_cast<const void*>(&dev::pa_logits_kernel<16>)
                   : num_heads == 32 ? reinterpret_cast<const void*>(&dev::pa_logits_kernel<32>)
                   : num_heads == 64 ? reinterpret_cast<const void*>(&dev::pa_logits_kernel<64>)
                                     : reinterpret_cast<const void*>(&dev::pa_logits_kernel<128>);
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
  if (e != cudaSuccess) return set_error(PA_ERR_CUDA, cudaGetErrorString(e));
  // Splits of a row block's tiles: enough CTAs for two waves over the SMs,
  // at most 128 tiles per CTA, at least 8 tiles per split.
  const int tiles = (num_kv + dev::kLgTile - 1) / dev::kLgTile;
  int splits = (2 * sms + nblk - 1) / nblk;
  splits = std::max(splits, (tiles + 127) / 128);
  splits = std::min(splits, std::max(1, tiles / 8));
  splits = std::max(1, std::min(splits, 65535));
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3((unsigned)nblk, (unsigned)splits, 1);
  cfg.blockDim = dim3((unsigned)dev::lg_threads(num_heads), 1, 1);
  cfg.dynamicSmemBytes = dev::kLgSmemBytes;
  cfg.stream = static_cast<cudaStream_t>(stream);
  void* args[] = {&p, &tmQ, &tmK};
  e = cudaLaunchKernelExC(&cfg, fn, args);
  if (e != cudaSuccess) return set_error(PA_ERR_CUDA, cudaGetErrorString(e));
  return PA_OK;
}
