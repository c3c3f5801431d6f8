// Shared definitions of the CUDA path (kernels and host launchers).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/mtpattn.h"

namespace mtpattn {

constexpr int kHeadDim = MTPATTN_HEAD_DIM;    // 256
constexpr int kPage = MTPATTN_PAGE_SIZE;      // 16 keys per page
constexpr int kMaxQLen = MTPATTN_MAX_Q_LEN;   // 4
constexpr int kMaxRows = 64;                  // q_len (<= 4) x ratio (<= 16) rows per CTA
constexpr float kLog2e = 1.4426950408889634f;

// Everything one call needs on the device.  Strides are in elements.
struct AttnParams {
  const __nv_bfloat16* q;
  int64_t q_stride_tok, q_stride_head;
  const uint8_t* k_cache;
  const uint8_t* v_cache;
  int64_t num_pages;
  const int32_t* block_tables;
  int32_t max_pages;
  const int32_t* seq_lens;
  const int32_t* cu_q;
  int32_t num_seqs, total_q, num_q_heads, num_kv_heads, ratio;
  const float* k_descale;
  const float* v_descale;
  float scale_log2;     // softmax_scale * log2(e): logits are kept in the log2 domain
  int32_t num_segments;
  int32_t slots_used;    // slots most rows use (<= num_segments): the reduce loads them with the LSEs
  uint32_t* tile_ctr;    // per-unit tile counters (workspace header; zero between calls)
  uint32_t* call_ctr;    // [2]: main-kernel CTAs started, finished (workspace header; both
                         // only grow, equal between calls): the reduce starts merging once
                         // every CTA of the main grid has counted itself out
  int32_t deterministic; // 1: fixed page ranges per piece (bit-identical repeats)
  int32_t scheduling;    // 0: chunks sized for max_pages, 1: pieces planned from the lengths
  float* o_part;        // [total_q * H_q][S][256] float32, normalised per segment
  float* lse_part;      // [total_q * H_q][S] float32, log2-sum-exp2 of the segment (NaN = error)
  // Slot pool (planned scheduling, when the caller left num_segments to the library): the
  // plan may give a long unit more than S pieces when short units use fewer.  The o_part
  // region then holds every unit's partials unit by unit, [row of the unit][piece], pool_cap
  // row-slots of 256 floats, followed by their LSEs (pool_lse, pool_cap floats); each output
  // row's first LSE slot holds kPoolMarker, the next two the row's first row-slot and its
  // number of pieces (as int32 bits).
  int32_t slot_pool;    // 1: the plan may use the pool layout
  int32_t pool_cap;     // row-slots of the pool: floor(rows * S * 256 / 257)
  float* pool_lse;      // o_part + pool_cap * 256
  __nv_bfloat16* out;
  int64_t out_stride_tok, out_stride_head;
  int32_t* status;      // optional
};

// Pages [begin, end) of segment s for a sequence of n_pages pages: equal shares of
// ceil(n_pages / S) pages, the tail segments possibly short or empty.
__host__ __device__ inline void segment_pages(int n_pages, int S, int s, int* begin, int* end) {
  int pps = (n_pages + S - 1) / S;
  int b = s * pps;
  int e = b + pps;
  if (b > n_pages) b = n_pages;
  if (e > n_pages) e = n_pages;
  *begin = b;
  *end = e;
}

// LSE bit pattern that marks an output row whose partials are in the slot pool (a NaN no
// arithmetic produces; the error NaN the kernels write is 0x7fc00000).
constexpr uint32_t kPoolMarker = 0x7fd00d1eu;

__device__ inline void set_status(int32_t* status, int bits) {
  if (status) atomicOr(status, bits);
}

// Host launchers (return cudaError_t of the launch).
// Workspace header: one tile counter per (sequence, KV head) unit, up to kMaxTileCounters
// units (beyond that the pieces keep fixed page ranges), zero on entry and on return; then
// the two call counters (AttnParams::call_ctr), equal on entry and on return.  Zero before
// the workspace's first use.
constexpr int kMaxTileCounters = 1024;
constexpr size_t kCallCtrOffset = kMaxTileCounters * sizeof(uint32_t);
constexpr size_t kWorkspaceHeaderBytes = kCallCtrOffset + 256;

// Planned scheduling handles at most this many (sequence, KV head) units (8 per lane of the
// planning warp), and no more units than SMs.
constexpr int kPlanUnits = 256;

// The main kernel: chunked scheduling (attn_main_tc.cu), or planned scheduling
// (attn_main_planned.cu) when p.scheduling asks for it and the batch allows it.
cudaError_t launch_attn_main(AttnParams& p, cudaStream_t stream);
cudaError_t launch_attn_main_planned(AttnParams& p, cudaStream_t stream);
cudaError_t launch_attn_reduce(const AttnParams& p, cudaStream_t stream);
// Tensor maps of the K and V caches (cached per cache, pool size and device).
bool kv_tensor_maps(const AttnParams& p, int device, CUtensorMap* mk, CUtensorMap* mv);
cudaError_t launch_stream_read(const void* buf, size_t bytes, uint32_t* sink, int blocks,
                               cudaStream_t stream);
int device_sm_count(int device);

}  // namespace mtpattn
