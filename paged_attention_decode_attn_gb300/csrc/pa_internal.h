// Internal definitions shared by the host side (plan, launch) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pa_decode.h"

namespace pa {

enum : int { kSchedBalanced = 1, kSchedPerUnit = 2 };
enum : int { kMergeDirect = 1, kMergeCluster = 2, kMergeLastArriver = 3, kMergeReducer = 4 };
enum : int { kScaleNone = 0, kScalePerTensor = 1, kScalePerToken = 2 };

// Device status bits (int32 in the workspace). kStatusScaleRange: a per-token
// V scale of a visible token outside [-2048, 2048] on the tensor-memory
// consumer (its FP16 V operand holds v * scale * 2^-4); that token's V is
// taken as zero.
enum : int { kStatusTimeout = 1, kStatusBadPage = 2, kStatusInternal = 4, kStatusScaleRange = 8 };

// Stage header flags.
enum : int { kSegFirst = 1, kSegLast = 2, kSegWhole = 4 };

constexpr int kMaxRows = 64;
constexpr int kCounterStride = 32;  // int32 per arrival counter: one 128-byte line

// Everything a tile/reducer launch needs, passed by value (__grid_constant__).
struct PaParams {
  // tensors
  uint16_t* out;              // BF16 [B*QL, Hq, D]
  const uint16_t* q;          // BF16 [B*QL, Hq, D]
  const int32_t* block_table; // [B, maxp]
  const int32_t* ctx_lens;    // [B]
  const float* k_scale;       // [1] or [num_pages, Hkv, S]
  const float* v_scale;
  const float* sinks;         // [Hq] or null
  const int32_t* topk_idx;    // [B, topk] or null
  float* part_o;              // [slots, Rpad, D]
  float* part_ml;             // [slots, Rpad, 2]  (max, sum) in log2 units
  int* counters;              // [U, kCounterStride]
  int4* unit_desc;            // [U] (nseg, s0, sbase, sstride) for the reducer
  int* status;                // device status word
  // shape
  int B, Hq, Hkv, G, QL, D, S, maxp, num_pages, R, Rpad;
  int window, causal, topk, has_sinks, scale_mode;
  float sm_scale_log2;  // sm_scale * log2(e)
  // schedule
  int sched, merge;
  int C;   // balanced: CTAs in the grid
  int seg_cost;  // balanced: virtual chunks charged per unit for its segment overhead
  int P;   // per-unit: partitions per unit
  int TT;  // tokens per stage (= chunk)
  int NS;  // ring stages
  int Wr, Wt, NCW;  // row warps, token warps, consumer warps
  int BH;           // rows per dense TMA box = min(S, TT)
  // dynamic shared memory layout (byte offsets from a 1024-aligned base)
  int off_stage, stage_bytes, off_scale;  // off_scale: within a stage
  int off_hdr, off_bar, off_merge, off_cpart, off_misc, off_pend, off_mml;
  int off_q, q_slot_bytes, NQ;  // Q ring: NQ (1 or 2) slots of Rpad rows x D BF16 values
  // tcgen05 consumer: 16-bit K and V operands (FP8 caches), Q and P operands,
  // the two MMA commit barriers, and the tensor-memory address slot
  int off_k16, off_v16, off_q16, off_p16, off_ubar, off_tslot, off_rows;
  int q_f16;  // queries and output are FP16 (else BF16)
  int v_tr;   // V cache in the transposed layout [pages, Hkv, S/8, D, 8] (BF16)
  // cache bases for the sparse row gathers (dense stages load through the tensor maps)
  const uint8_t* k_cache;
  const uint8_t* v_cache;
};

// Host-visible shared-memory sizing for a kernel configuration.
struct SmemLayout {
  int stage_bytes, off_stage, off_scale, off_hdr, off_bar, off_merge, off_cpart, off_misc, off_pend, off_mml;
  int off_q, q_slot_bytes, nq, off_k16, off_v16, off_q16, off_p16, off_ubar, off_tslot, off_rows, total;
};

using KernelFn = void (*)(PaParams, CUtensorMap, CUtensorMap);

// Tile-kernel instantiations (defined in the pa_tile_*.cu files).
// Returns null when the combination is not instantiated.
const void* tile_kernel_fp8_d128(int vtok, int wide);
const void* tile_kernel_fp4_d128(int wide);
const void* tile_kernel_fp8_d256(int vtok);
const void* tile_kernel_bf16(int d, int wide, int q_f16);
const void* tile_kernel_bf16_q16(int d, int wide);
const void* tile_kernel_bf16_tv(int d, int wide, int q_f16);
const void* tile_kernel_bf16_tv_q16(int d, int wide);
const void* reduce_kernel(int d);
// Tensor-memory consumer instantiations (FP8 head_dim 128/256, BF16 head_dim
// 128; rh = query rows per softmax warpgroup, 16 or 32; nwg = softmax
// warpgroups, 2 or 4).
const void* mtp_kernel(int fp8, int d, int vtok, int rh, int nwg);

}  // namespace pa

struct pa_plan;

namespace pa {

// Makes `device` current for the guard's lifetime and restores the caller's
// current device on every return path.
class DeviceGuard {
 public:
  explicit DeviceGuard(int device) {
    err_ = cudaGetDevice(&prev_);
    if (err_ == cudaSuccess && prev_ != device) {
      err_ = cudaSetDevice(device);
      switched_ = err_ == cudaSuccess;
    }
  }
  ~DeviceGuard() {
    if (switched_) (void)cudaSetDevice(prev_);
  }
  cudaError_t error() const { return err_; }

 private:
  int prev_ = 0;
  bool switched_ = false;
  cudaError_t err_ = cudaSuccess;
};

// Host helpers shared with the no-allocation entry point (pa_noalloc.cu).
pa_status launch_on_workspace(const pa_plan* plan, void* ws, size_t ws_bytes, void* out, const void* q,
                              const void* k_cache, const void* v_cache, const int32_t* block_table,
                              const int32_t* ctx_lens, const float* k_scale, const float* v_scale, int window,
                              const float* sinks, void* stream);
size_t plan_workspace_layout(const pa_plan* plan, size_t* zero_from, int* device, int* sparse);
pa_status set_error(pa_status status, const char* message);

}  // namespace pa
