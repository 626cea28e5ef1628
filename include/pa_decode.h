/*
 * pa_decode.h — C ABI of the GB300 (sm_103a) paged-attention decode library.
 *
 * What the library computes
 * -------------------------
 * For every sequence b, query index i in [0, query_len), query head h and its
 * KV head g = h / (num_q_heads / num_kv_heads), the BF16 output row
 *
 *     out[b*QL + i, h, :] = sum_t softmax_t(x) * v_t      (t in the visible set)
 *     x_t = sm_scale * <q[b*QL + i, h, :], k_t>
 *
 * over a KV cache split into fixed-size pages that a per-sequence int32 block
 * table addresses (PR "Add paged-attention Tile kernel": pa_decode(output,
 * query, key_cache, value_cache, block_tables, context_lengths, key_scale,
 * value_scale, ...) and its shape checks). The visible set of row (b, i) is
 * t in [0, L_b) with, for causal multi-token (MTP) queries, t <= p and, for a
 * sliding window W > 0, t > p - W, where p = L_b - QL + i (PR "Extend packed
 * D256 PA decode pipe to page16, transposed V and sliding windows": windows
 * 0/1/17/257/8193, QL 1-4). Optional per-query-head sink logits add e^(s - m)
 * to the softmax denominator only (PR "Merge gfx1250 PA decode partitions in
 * the tile kernel and speed up dense decode": sinks keep a merge path). An
 * empty visible set gives a zero row.
 *
 * The KV range is split into partitions whose online-softmax partials
 * (running max, running sum, unnormalised output) are merged in partition
 * order, inside a thread-block cluster over distributed shared memory, by the
 * last-arriving CTA through device-scope arrival counters, or by a standalone
 * reducer kernel (same PR, "Partition merges"). All merge mechanisms use the
 * same arithmetic in the same order, so for one plan schedule they give
 * bit-identical outputs.
 *
 * Layouts (all tensors are caller-owned device memory, row-major, contiguous)
 * --------------------------------------------------------------------------
 *   q, out        [batch*query_len, num_q_heads, head_dim]     BF16 or FP16
 *                 (the plan's q_dtype)
 *   k_cache,
 *   v_cache       [num_pages, num_kv_heads, page_size, head_dim]
 *                 FP8 e4m3fn bytes (OCP) or BF16; MXFP4:
 *                 [num_pages, num_kv_heads, page_size, head_dim / 2] bytes,
 *                 two E2M1 codes each (see PA_KV_MXFP4); v_cache with
 *                 PA_V_TRANSPOSED: [num_pages, num_kv_heads, page_size / 8,
 *                 head_dim, 8] BF16
 *   block_table   [batch, max_pages_per_seq]  int32 physical page ids; only
 *                 the entries covering [0, L_b) are ever read
 *   ctx_lens      [batch]  int32, 0 <= L_b <= max_pages_per_seq * page_size
 *   k_scale,
 *   v_scale       float32 [1] (per tensor) or [num_pages, num_kv_heads,
 *                 page_size] (per token); NULL when scale_mode is NONE;
 *                 MXFP4: uint8 E8M0 [num_pages, num_kv_heads, page_size,
 *                 head_dim / 32] (passed through the float pointer)
 *   sinks         float32 [num_q_heads] (natural-log units, not multiplied
 *                 by sm_scale) or NULL
 *   topk_idx      int32 [batch, sparse_topk] logical token positions;
 *                 entries outside [0, L_b) are ignored (sparse decode only)
 * Every pointer must be 16-byte aligned.
 *
 * Errors and ownership
 * --------------------
 * Functions return a pa_status; on failure a thread-local message is
 * available from pa_last_error(). Nothing aborts. pa_decode* allocates no
 * memory, never synchronises the stream and launches only on the given
 * stream, so calls can be captured in a CUDA graph. The plan owns host
 * metadata only; its workspace (partials, arrival counters, a device status
 * word) is caller-allocated device memory, bound once with
 * pa_plan_set_workspace and zero-filled by the caller before first use.
 * Arrival counters reset themselves, so the workspace needs no clearing
 * between calls. A plan (its workspace) must not be used by two decodes that
 * can run concurrently.
 */
#ifndef PA_DECODE_H
#define PA_DECODE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PA_API __attribute__((visibility("default")))
#else
#define PA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pa_status {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size or shape */
  PA_ERR_UNSUPPORTED = 2,  /* valid but not implemented (head_dim, rows, ...) */
  PA_ERR_WORKSPACE = 3,    /* workspace missing or too small */
  PA_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed */
  PA_ERR_DEVICE_STATUS = 5 /* a kernel reported a timeout in its status word */
} pa_status;

/* KV cache element types. MXFP4 (PR "Merge gfx1250 PA decode partitions in
 * the tile kernel and speed up dense decode", merge-resolution notes, names
 * MXFP4 K/V; the layout is this library's reading of the OCP Microscaling
 * (MX) v1.0 format): each K/V token row of head_dim (128) values is
 * head_dim / 2 bytes of FP4 E2M1 codes, element d in the low nibble of byte
 * d / 2 when d is even and in the high nibble when odd; its head_dim / 32 E8M0
 * block scales (value 2^(code - 127)) are the bytes
 * scale[((page * num_kv_heads + kv_head) * page_size + slot) * head_dim / 32 + d / 32],
 * passed through the k_scale / v_scale arguments. */
enum { PA_KV_FP8_E4M3 = 0, PA_KV_BF16 = 1, PA_KV_MXFP4 = 2 };
/* Element type of the queries and of the output (PR "Extend packed D256 PA
 * decode pipe to page16, transposed V and sliding windows", Validation, and PR
 * "Merge gfx1250 PA decode partitions in the tile kernel and speed up dense
 * decode", Validation, run BF16 and FP16 queries). */
enum { PA_Q_BF16 = 0, PA_Q_FP16 = 1 };
/* Layout of the V cache (PR "Extend packed D256 PA decode pipe to page16,
 * transposed V and sliding windows", and PR "Merge gfx1250 PA decode
 * partitions in the tile kernel and speed up dense decode", where transposed
 * V "spaces its eight-token chunks 16 * head_dim bytes apart"): PA_V_PLAIN is
 * [num_pages, num_kv_heads, page_size, head_dim]; PA_V_TRANSPOSED (BF16 caches,
 * dense decode, the tile consumer) is [num_pages, num_kv_heads, page_size / 8,
 * head_dim, 8]: for each chunk of 8 consecutive tokens, the 8 values of one
 * head dim are contiguous. */
enum { PA_V_PLAIN = 0, PA_V_TRANSPOSED = 1 };
/* PA_SCALE_MX_BLOCK: the E8M0 block scales of MXFP4 caches (required by them,
 * accepted by no other cache type). */
enum { PA_SCALE_NONE = 0, PA_SCALE_PER_TENSOR = 1, PA_SCALE_PER_TOKEN = 2, PA_SCALE_MX_BLOCK = 3 };

/* How partitions of one (sequence, KV head) are merged. */
enum {
  PA_MERGE_AUTO = 0,
  PA_MERGE_DIRECT = 1,       /* one partition per unit: the tile writes output */
  PA_MERGE_CLUSTER = 2,      /* P in [2, 16] CTAs of a cluster merge over DSMEM */
  PA_MERGE_LAST_ARRIVER = 3, /* the last CTA to arrive on a unit merges it */
  PA_MERGE_REDUCER = 4       /* a second kernel merges the partials */
};

/* How a stage is consumed. The tile consumer runs mma.sync per 8-row warp
 * (any shape, every cache format and V layout); the tensor-memory consumer
 * issues tcgen05.mma from a dedicated warp with accumulators in TMEM, two or
 * four softmax warpgroups splitting the rows (dense decode with 17..64 rows
 * per KV head, FP8 head_dim 128/256 or BF16 head_dim 128 with BF16 queries
 * and plain V; head_dim 256 with 9..32 rows; no MXFP4). AUTO takes the
 * tensor-memory consumer wherever it covers the shape (measured faster on
 * every such shape), else the tile consumer. */
enum { PA_CONSUMER_AUTO = 0, PA_CONSUMER_TILE = 1, PA_CONSUMER_TMEM = 2 };

/* How KV chunks are assigned to CTAs. */
enum {
  PA_SCHED_AUTO = 0,
  PA_SCHED_BALANCED = 1, /* all units' chunks split evenly over a persistent grid */
  PA_SCHED_PER_UNIT = 2  /* P CTAs per (sequence, KV head), P = partitions */
};

typedef struct pa_plan_desc {
  int batch;
  int num_q_heads;
  int num_kv_heads;      /* num_q_heads % num_kv_heads == 0 */
  int head_dim;          /* 128 or 256; 64 with BF16 caches; MXFP4: 128 (PA_ERR_UNSUPPORTED otherwise) */
  int query_len;         /* >= 1 (MTP rows); rows = query_len * group <= 64 (32 at head_dim 256) */
  int page_size;         /* 16, 32, 64, 128 or 256 tokens */
  int max_pages_per_seq; /* block-table row stride (int32 elements) */
  int num_pages;         /* pages in the cache pool */
  int max_context_len;   /* host bound used for automatic choices; 0 = unknown */
  int kv_dtype;          /* PA_KV_* */
  int scale_mode;        /* PA_SCALE_* (FP8: NONE/PER_TENSOR/PER_TOKEN; BF16: NONE; MXFP4: MX_BLOCK) */
  int causal;            /* causal mask among the query_len new tokens */
  int has_sinks;
  int sparse_topk;       /* 0 = dense decode; > 0 = index-list decode (query_len 1) */
  float sm_scale;        /* 0 => 1/sqrt(head_dim); must be > 0 otherwise */
  int max_partitions;    /* per-unit schedule partitions; 0 => automatic */
  int merge_mode;        /* PA_MERGE_* */
  int schedule;          /* PA_SCHED_* */
  int sm_count_override; /* 0 => device attribute (tests: simulated SM counts) */
  int ctas_per_sm_override; /* 0 => occupancy query */
  int device;            /* CUDA device ordinal the plan is for */
  int consumer;          /* PA_CONSUMER_*; TMEM on an unsupported shape is PA_ERR_UNSUPPORTED */
  int q_dtype;           /* PA_Q_*: element type of q and out (0 = BF16) */
  int v_layout;          /* PA_V_*: layout of v_cache (0 = plain) */
} pa_plan_desc;

typedef struct pa_plan_info {
  int merge_mode;      /* resolved PA_MERGE_* */
  int schedule;        /* resolved PA_SCHED_* */
  int num_partitions;  /* per-unit schedule: P; balanced: 0 */
  int stage_tokens;    /* tokens per ring stage (= chunk granularity) */
  int num_stages;      /* shared-memory ring depth */
  int rows;            /* query rows per (sequence, KV head) = group * query_len */
  int rows_per_warp;   /* 8 or 16 */
  int row_warps;       /* consumer warps splitting the rows */
  int token_warps;     /* consumer warps splitting each stage's tokens */
  int block_threads;   /* consumer warps * 32 + one producer warp */
  int grid;            /* CTAs of the tile kernel */
  int cluster;         /* cluster size (1 = none) */
  int ctas_per_sm;
  int sm_count;
  int launches_per_call;
  int units;           /* batch * num_kv_heads */
  int consumer;        /* resolved PA_CONSUMER_* */
  size_t smem_bytes;   /* dynamic shared memory of the tile kernel */
  size_t workspace_bytes;
  size_t partial_slots;
  size_t status_offset; /* byte offset of the int32 device status word */
} pa_plan_info;

typedef struct pa_plan pa_plan_t;

/* Validate desc, size partitions from the SM count and occupancy, pick the
 * merge mechanism. Follows PR "Add paged-attention Tile kernel" (the
 * per-sequence plan limit defaults to the device's compute-unit count; head
 * dimension and shape checks reject what the kernels cannot run) and PR "Merge
 * gfx1250 PA decode partitions in the tile kernel and speed up dense decode",
 * Partition merges (cluster merge for 2..16 partitions, last-arriver merge
 * for one-slot plans, the reducer otherwise).
 * desc: read only, not retained. out: receives a host-heap plan owned by the
 * caller (release with pa_plan_destroy); set to NULL on failure.
 * Errors: PA_ERR_INVALID_ARG (bad field), PA_ERR_UNSUPPORTED (valid but not
 * built: head_dim, rows, page size), PA_ERR_CUDA (device attribute or
 * occupancy query failed). Host only: with both overrides set it touches no
 * device; otherwise it queries the plan's device and restores the caller's
 * current device before returning. */
PA_API pa_status pa_plan_create(const pa_plan_desc* desc, pa_plan_t** out);

/* Bytes of caller-owned device workspace the plan needs: partial (max, sum,
 * unnormalised output) per split segment (PR "Add paged-attention Tile
 * kernel": exp_sums, max_logits and tmp_output of a partitioned call), arrival
 * counters at one 128-byte line each (PR "Merge gfx1250 PA decode partitions
 * in the tile kernel and speed up dense decode", Partition merges:
 * [batch, kv_heads, 32] int32), reducer descriptors and the status word.
 * Returns 0 for a NULL plan. */
PA_API size_t pa_plan_workspace_bytes(const pa_plan_t* plan);

/* Bind zero-filled device memory of at least pa_plan_workspace_bytes bytes
 * (256-byte aligned) on the plan's device. The plan does not take ownership;
 * the memory must outlive every decode enqueued with the plan. The arrival
 * counters in it are zeroed once here by the caller and reset by their last
 * arrival afterwards (PR "Merge gfx1250 PA decode partitions in the tile
 * kernel and speed up dense decode", Partition merges), so CUDA-graph replays
 * need no host work. Errors: PA_ERR_INVALID_ARG (NULL plan), PA_ERR_WORKSPACE
 * (NULL, misaligned or too small). */
PA_API pa_status pa_plan_set_workspace(pa_plan_t* plan, void* dev_ptr, size_t bytes);

/* Copy the resolved plan (partitions, stage size, merge mode, grid,
 * workspace layout) into *info, for tests that check the sizing rule of PR
 * "Add paged-attention Tile kernel" (partition count from the compute-unit
 * count) bit for bit. Errors: PA_ERR_INVALID_ARG for NULL arguments. */
PA_API pa_status pa_plan_get_info(const pa_plan_t* plan, pa_plan_info* info);

/* Free a plan (NULL is a no-op). Decodes already enqueued with it are not
 * affected: they carry their arguments by value. */
PA_API void pa_plan_destroy(pa_plan_t* plan);

/* Dense paged decode of one batch on `stream` (a cudaStream_t; NULL = legacy
 * default stream): PR "Add paged-attention Tile kernel" (pa_decode(output,
 * query, key_cache, value_cache, block_tables, context_lengths, key_scale,
 * value_scale, ...)), with the sliding window and sinks of PR "Extend packed
 * D256 PA decode pipe to page16, transposed V and sliding windows" and PR
 * "Merge gfx1250 PA decode partitions in the tile kernel and speed up dense
 * decode". q and out: device [batch * query_len, num_q_heads, head_dim]
 * elements of the plan's q_dtype (BF16 or FP16), row-major; out is written
 * in that type. window: 0 = off, else W >= 1 (requires causal or query_len 1).
 * Scales: required (device float32) when the plan's scale_mode is not NONE.
 * Errors: PA_ERR_INVALID_ARG (NULL or misaligned pointer, negative window,
 * sparse plan), PA_ERR_UNSUPPORTED (window with non-causal multi-token
 * queries), PA_ERR_WORKSPACE (none bound), PA_ERR_CUDA (launch failed).
 * Returns after enqueueing; a page id outside [0, num_pages) or a bounded
 * wait that ran out sets a bit in the device status word
 * (pa_plan_info.status_offset inside the workspace). */
PA_API pa_status pa_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* block_table, const int32_t* ctx_lens, const float* k_scale,
                    const float* v_scale, int window, const float* sinks, const pa_plan_t* plan,
                    void* stream);

/* Sparse (top-k index list) decode: each sequence (query_len 1) attends to
 * the tokens its row of topk_idx lists, gathered through the block table (PR
 * "Merge gfx1250 PA decode partitions in the tile kernel and speed up dense
 * decode": sparse decode over 2048 top-k page16 tokens per row, and sparse
 * prefill, where row r lists min(r + 1, 2048) tokens and the remaining entries
 * are ignored). No causal mask or window; entries outside [0, L_b) are skipped.
 * Errors as pa_decode, plus PA_ERR_INVALID_ARG for a dense plan or a NULL
 * topk_idx. */
PA_API pa_status pa_decode_sparse(void* out, const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* block_table, const int32_t* ctx_lens,
                           const int32_t* topk_idx, const float* k_scale, const float* v_scale,
                           const float* sinks, const pa_plan_t* plan, void* stream);

/* Dense decode exactly like pa_decode, but on a scratch buffer built into the
 * library instead of the plan's workspace, so it needs no device allocation
 * from the caller (for code that cannot call cudaMalloc: plugins inside a
 * framework that owns all device memory, or latency-critical paths where an
 * allocation may synchronise the device). The reference pages have no
 * counterpart to this entry point. The scratch is 32 MiB per GPU that loads
 * the library, held until the process exits; plans whose
 * pa_plan_workspace_bytes exceed it get PA_ERR_WORKSPACE. No workspace needs
 * to be bound to the plan. The first call on a device looks up the scratch
 * address (cudaGetSymbolAddress); make that first call before any stream
 * capture. Every call shares the one buffer: calls that can overlap on the
 * GPU race, so serialise them. Each call zeroes the scratch's counters and
 * status word on `stream` before its kernel. The device status word lives in
 * that private scratch, so on this path a page id out of range or a bounded
 * wait that ran out is not reported to the caller (pa_decode reports both
 * through the workspace's status word); a caller that needs that check
 * should use pa_decode. */
PA_API pa_status pa_decode_noalloc(void* out, const void* q, const void* k_cache, const void* v_cache,
                                   const int32_t* block_table, const int32_t* ctx_lens, const float* k_scale,
                                   const float* v_scale, int window, const float* sinks, const pa_plan_t* plan,
                                   void* stream);

/* Indexer logits: the scoring step upstream of sparse decode, which ranks KV
 * tokens for each query row (PR "[FlyDSL] fp8_mqa_logits gfx942: add
 * LDS-staged variant, use it by default": FP8 Q and KV, a ReLU x weight
 * epilogue reduced over the heads, per-row KV windows, and -inf written
 * outside them by the kernel itself when clean_logits is set). For query row
 * r and KV token j in its window [ks[r], ke[r]) (clipped to [0, num_kv)):
 *
 *   logits[r * logits_stride + j] =
 *       sum_h weights[r * num_heads + h] * max(0, kv_scale[j] * sum_d q[r][h][d] * kv[j][d])
 *
 * with q and kv decoded exactly from OCP e4m3fn bytes; every other j in
 * [0, num_kv) is set to -inf when clean_logits != 0 and left untouched
 * otherwise. Arguments (device memory, 16-byte aligned, caller-owned):
 *   logits   float32 [rows, logits_stride] (logits_stride >= num_kv, a multiple of 4)
 *   q        e4m3 bytes [rows, num_heads, head_dim]
 *   kv       e4m3 bytes [num_kv, head_dim]
 *   kv_scale float32 [num_kv], >= 0 (the per-token dequantisation scale)
 *   weights  float32 [rows, num_heads] (any head weighting, softmax scale included)
 *   ks, ke   int32 [rows] window bounds
 *   status   int32 device word or NULL: a bounded wait that ran out sets a bit
 * num_heads: 16, 32, 64 or 128; head_dim: 128. One kernel launch on `stream`
 * (tcgen05 FP8 MMAs, FP32 accumulation); nothing is allocated.
 * Errors: PA_ERR_INVALID_ARG (null or misaligned pointer, bad size),
 * PA_ERR_UNSUPPORTED (head count or head_dim), PA_ERR_CUDA (launch). */
PA_API pa_status pa_mqa_logits(float* logits, int logits_stride, const void* q, const void* kv,
                               const float* kv_scale, const float* weights, const int32_t* ks,
                               const int32_t* ke, int rows, int num_heads, int head_dim, int num_kv,
                               int clean_logits, int32_t* status, int device, void* stream);

PA_API const char* pa_strerror(pa_status status);

/* Message of the last failure on this thread ("" if none). */
PA_API const char* pa_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_DECODE_H */
