// C-ABI entry points: argument checks, the segment heuristic, workspace
// carving and the two launches.  Everything here runs on the host and never
// touches device memory contents, so a call can be captured in a CUDA graph.
#include "common.cuh"

#include <algorithm>
#include <atomic>
#include <climits>

#include <math.h>
#include <stddef.h>

namespace mtpattn {

// The planned main kernel with Q and P rounded to single e4m3 codes (attn_main_planned_qp8.cu,
// where the common declaration of launch_attn_main_planned takes this name); planned
// scheduling only, so the caller checks that the batch allows it.
cudaError_t launch_attn_main_planned_qp8(AttnParams& p, cudaStream_t stream);

int device_sm_count(int device) {
  // Filled on first use per device; atomics, since calls may come from several host threads.
  static std::atomic<int> cache[64];
  if (device < 0) {
    if (cudaGetDevice(&device) != cudaSuccess) return -1;
  }
  if (device >= 64) return -1;
  const int cached = cache[device].load(std::memory_order_relaxed);
  if (cached > 0) return cached;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
      sms <= 0) {
    cudaGetLastError();
    return -1;
  }
  cache[device].store(sms, std::memory_order_relaxed);
  return sms;
}

namespace {

std::atomic<int> g_deterministic{0};   // scheduling switch, see mtp_verify_attn_set_deterministic
std::atomic<int> g_scheduling{MTPATTN_SCHED_PLANNED};   // see mtp_verify_attn_set_scheduling

constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// A pointer the kernels may dereference: device (or managed) memory of `device`.
bool on_device(const void* ptr, int device) {
  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, ptr) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged) return false;
  return attr.device == device;
}

}  // namespace
}  // namespace mtpattn

using namespace mtpattn;

extern "C" int32_t mtp_verify_attn_num_segments(int32_t num_seqs, int32_t num_kv_heads,
                                                int32_t max_pages_per_seq, int32_t device) {
  if (num_seqs <= 0 || num_kv_heads <= 0 || max_pages_per_seq <= 0) return MTPATTN_E_ARG;
  const int sms = device_sm_count(device);
  if (sms <= 0) return MTPATTN_E_DEVICE;
  const long long units = static_cast<long long>(num_seqs) * num_kv_heads;
  if (g_scheduling.load(std::memory_order_relaxed) == MTPATTN_SCHED_PLANNED && units <= kPlanUnits &&
      units <= sms) {
    // Planned scheduling sizes the pieces from the lengths, so S only caps the pieces of one
    // unit: allow a single long sequence every SM the other units leave (one each), but no
    // piece shorter than one 128-key tile.
    long long s = std::min<long long>(sms - units + 1, (max_pages_per_seq + 7) / 8);
    if (s < 1) s = 1;
    if (s > MTPATTN_MAX_SEGMENTS) s = MTPATTN_MAX_SEGMENTS;
    return static_cast<int32_t>(s);
  }
  // Chunked scheduling: enough split slots for a unit of max_pages_per_seq pages to be cut at
  // every boundary of an equal per-SM share of the batch's pages.
  const long long V = max_pages_per_seq;
  const long long total = static_cast<long long>(num_seqs) * num_kv_heads * V;
  const long long share = (total + sms - 1) / sms;
  long long s = (V + share - 1) / share + 1;
  if (s > MTPATTN_MAX_SEGMENTS) s = MTPATTN_MAX_SEGMENTS;
  return static_cast<int32_t>(s);
}

extern "C" size_t mtp_verify_attn_workspace_size(int32_t total_q, int32_t num_q_heads,
                                                 int32_t num_segments) {
  if (total_q < 0 || num_q_heads <= 0 || num_segments < 1 ||
      num_segments > MTPATTN_MAX_SEGMENTS)
    return 0;
  const size_t rows = static_cast<size_t>(total_q) * num_q_heads;
  const size_t lse = align_up(rows * num_segments * sizeof(float));
  const size_t o = align_up(rows * num_segments * kHeadDim * sizeof(float));
  return kWorkspaceHeaderBytes + lse + o;
}

namespace {

// The two precision tiers share every check and the launch set-up; qp_fp8 selects the
// kernel that rounds Q and P to single e4m3 codes (planned scheduling only).
int verify_fwd(const void* q, int64_t q_stride_tok, int64_t q_stride_head, const void* k_cache,
               const void* v_cache, int64_t num_pages, const int32_t* block_tables,
               int32_t max_pages_per_seq, const int32_t* seq_lens, const int32_t* cu_seqlens_q,
               int32_t num_seqs, int32_t total_q, int32_t num_q_heads, int32_t num_kv_heads,
               const float* k_descale, const float* v_descale, float softmax_scale,
               int32_t num_segments, void* workspace, size_t workspace_bytes, void* out,
               int64_t out_stride_tok, int64_t out_stride_head, int32_t* status, void* stream,
               bool qp_fp8) {
  // 1. plain argument checks
  if (num_seqs < 0 || total_q < 0 || num_pages < 0 || max_pages_per_seq < 0 ||
      num_q_heads <= 0 || num_kv_heads <= 0)
    return MTPATTN_E_ARG;
  if (num_seqs == 0) return total_q == 0 ? MTPATTN_OK : MTPATTN_E_ARG;
  if (total_q < num_seqs) return MTPATTN_E_ARG;          // every sequence has >= 1 query token
  if (!q || !k_cache || !v_cache || !block_tables || !seq_lens || !cu_seqlens_q ||
      !k_descale || !v_descale || !out || num_pages == 0 || max_pages_per_seq == 0)
    return MTPATTN_E_ARG;
  if (!isfinite(softmax_scale)) return MTPATTN_E_ARG;
  if (q_stride_tok <= 0 || q_stride_head <= 0 || out_stride_tok <= 0 || out_stride_head <= 0 ||
      (q_stride_tok | q_stride_head | out_stride_tok | out_stride_head) % 8 != 0)
    return MTPATTN_E_ARG;
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(block_tables, 4) || !aligned(seq_lens, 4) || !aligned(cu_seqlens_q, 4) ||
      !aligned(k_descale, 4) || !aligned(v_descale, 4) || !aligned(status, 4))
    return MTPATTN_E_ARG;
  // 2. the supported envelope
  if (num_q_heads % num_kv_heads) return MTPATTN_E_UNSUPPORTED;
  const int ratio = num_q_heads / num_kv_heads;
  if (ratio != 8 && ratio != 16) return MTPATTN_E_UNSUPPORTED;
  if (total_q > static_cast<int64_t>(num_seqs) * MTPATTN_MAX_Q_LEN) return MTPATTN_E_UNSUPPORTED;
  if (num_segments < 0 || num_segments > MTPATTN_MAX_SEGMENTS) return MTPATTN_E_UNSUPPORTED;
  // 3. the segment count (the heuristic needs the device) and the workspace
  int device = -1;
  const bool library_chose_s = num_segments == 0;
  if (num_segments == 0) {
    if (cudaGetDevice(&device) != cudaSuccess) {
      cudaGetLastError();
      return MTPATTN_E_DEVICE;
    }
    num_segments = mtp_verify_attn_num_segments(num_seqs, num_kv_heads, max_pages_per_seq, device);
    if (num_segments < 1) return MTPATTN_E_DEVICE;
  }
  const size_t need = mtp_verify_attn_workspace_size(total_q, num_q_heads, num_segments);
  if (!workspace || !aligned(workspace, kAlign) || workspace_bytes < need)
    return MTPATTN_E_WORKSPACE;
  if (qp_fp8) {                  // the fp8 tier exists for planned scheduling only
    const int sms = device_sm_count(-1);
    if (sms <= 0) return MTPATTN_E_DEVICE;
    const int64_t units = static_cast<int64_t>(num_seqs) * num_kv_heads;
    if (units > kPlanUnits || units > sms) return MTPATTN_E_UNSUPPORTED;
  }
  // 4. every pointer must be memory the kernels can read on the current device
  if (device < 0 && cudaGetDevice(&device) != cudaSuccess) {
    cudaGetLastError();
    return MTPATTN_E_DEVICE;
  }
  const void* ptrs[] = {q, k_cache, v_cache, block_tables, seq_lens, cu_seqlens_q,
                        k_descale, v_descale, workspace, out};
  for (const void* ptr : ptrs)
    if (!on_device(ptr, device)) return MTPATTN_E_DEVICE;
  if (status && !on_device(status, device)) return MTPATTN_E_DEVICE;

  AttnParams p;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.q_stride_tok = q_stride_tok;
  p.q_stride_head = q_stride_head;
  p.k_cache = static_cast<const uint8_t*>(k_cache);
  p.v_cache = static_cast<const uint8_t*>(v_cache);
  p.num_pages = num_pages;
  p.block_tables = block_tables;
  p.max_pages = max_pages_per_seq;
  p.seq_lens = seq_lens;
  p.cu_q = cu_seqlens_q;
  p.num_seqs = num_seqs;
  p.total_q = total_q;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = num_kv_heads;
  p.ratio = ratio;
  p.k_descale = k_descale;
  p.v_descale = v_descale;
  p.scale_log2 = softmax_scale * kLog2e;
  p.num_segments = num_segments;
  p.slots_used = num_segments;
  const size_t rows = static_cast<size_t>(total_q) * num_q_heads;
  // The slot pool (planned scheduling only): when the library chose S, a long unit may take
  // more than S pieces if short units use fewer, inside the same rows x S partial slots.
  p.slot_pool = (library_chose_s && num_segments >= 3) ? 1 : 0;
  {
    const int64_t cap = static_cast<int64_t>(rows) * num_segments * kHeadDim / (kHeadDim + 1);
    p.pool_cap = static_cast<int32_t>(std::min<int64_t>(cap, INT32_MAX / kHeadDim));
  }
  p.tile_ctr = static_cast<uint32_t*>(workspace);
  p.call_ctr = reinterpret_cast<uint32_t*>(static_cast<char*>(workspace) + kCallCtrOffset);
  p.lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + kWorkspaceHeaderBytes);
  p.o_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + kWorkspaceHeaderBytes +
                                      align_up(rows * num_segments * sizeof(float)));
  p.pool_lse = p.o_part + static_cast<int64_t>(p.pool_cap) * kHeadDim;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.out_stride_tok = out_stride_tok;
  p.out_stride_head = out_stride_head;
  p.status = status;
  p.deterministic = g_deterministic.load(std::memory_order_relaxed);
  p.scheduling = qp_fp8 ? MTPATTN_SCHED_PLANNED : g_scheduling.load(std::memory_order_relaxed);

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if ((qp_fp8 ? launch_attn_main_planned_qp8(p, st) : launch_attn_main(p, st)) != cudaSuccess)
    return MTPATTN_E_LAUNCH;
  if (launch_attn_reduce(p, st) != cudaSuccess) return MTPATTN_E_LAUNCH;
  return MTPATTN_OK;
}

}  // namespace

extern "C" int mtp_verify_attn_fwd(const void* q, int64_t q_stride_tok, int64_t q_stride_head,
                                   const void* k_cache, const void* v_cache, int64_t num_pages,
                                   const int32_t* block_tables, int32_t max_pages_per_seq,
                                   const int32_t* seq_lens, const int32_t* cu_seqlens_q,
                                   int32_t num_seqs, int32_t total_q, int32_t num_q_heads,
                                   int32_t num_kv_heads, const float* k_descale,
                                   const float* v_descale, float softmax_scale,
                                   int32_t num_segments, void* workspace,
                                   size_t workspace_bytes, void* out, int64_t out_stride_tok,
                                   int64_t out_stride_head, int32_t* status, void* stream) {
  return verify_fwd(q, q_stride_tok, q_stride_head, k_cache, v_cache, num_pages, block_tables,
                    max_pages_per_seq, seq_lens, cu_seqlens_q, num_seqs, total_q, num_q_heads,
                    num_kv_heads, k_descale, v_descale, softmax_scale, num_segments, workspace,
                    workspace_bytes, out, out_stride_tok, out_stride_head, status, stream, false);
}

extern "C" int mtp_verify_attn_fwd_qp_fp8(const void* q, int64_t q_stride_tok,
                                          int64_t q_stride_head, const void* k_cache,
                                          const void* v_cache, int64_t num_pages,
                                          const int32_t* block_tables, int32_t max_pages_per_seq,
                                          const int32_t* seq_lens, const int32_t* cu_seqlens_q,
                                          int32_t num_seqs, int32_t total_q, int32_t num_q_heads,
                                          int32_t num_kv_heads, const float* k_descale,
                                          const float* v_descale, float softmax_scale,
                                          int32_t num_segments, void* workspace,
                                          size_t workspace_bytes, void* out,
                                          int64_t out_stride_tok, int64_t out_stride_head,
                                          int32_t* status, void* stream) {
  return verify_fwd(q, q_stride_tok, q_stride_head, k_cache, v_cache, num_pages, block_tables,
                    max_pages_per_seq, seq_lens, cu_seqlens_q, num_seqs, total_q, num_q_heads,
                    num_kv_heads, k_descale, v_descale, softmax_scale, num_segments, workspace,
                    workspace_bytes, out, out_stride_tok, out_stride_head, status, stream, true);
}

extern "C" void mtp_verify_attn_set_deterministic(int32_t on) { g_deterministic.store(on ? 1 : 0); }
extern "C" int32_t mtp_verify_attn_get_deterministic(void) { return g_deterministic.load(); }
extern "C" int32_t mtp_verify_attn_set_scheduling(int32_t mode) {
  if (mode != MTPATTN_SCHED_CHUNKED && mode != MTPATTN_SCHED_PLANNED) return MTPATTN_E_ARG;
  g_scheduling.store(mode);
  return MTPATTN_OK;
}
extern "C" int32_t mtp_verify_attn_get_scheduling(void) { return g_scheduling.load(); }

extern "C" const char* mtp_verify_attn_strerror(int status) {
  switch (status) {
    case MTPATTN_OK: return "ok";
    case MTPATTN_E_ARG: return "invalid argument (null pointer, negative count, stride or alignment)";
    case MTPATTN_E_UNSUPPORTED: return "unsupported configuration (GQA ratio must be 8 or 16, q_len <= 4, num_segments in [0, 64])";
    case MTPATTN_E_DEVICE: return "pointer is not device memory of the current CUDA device, or no CUDA device";
    case MTPATTN_E_WORKSPACE: return "workspace missing, smaller than mtp_verify_attn_workspace_size() or not 256-byte aligned";
    case MTPATTN_E_LAUNCH: return "kernel launch failed";
    case MTPATTN_E_SCRATCH_LIMIT: return "the call needs more scratch than the library's static array (MTPATTN_STATIC_SCRATCH_BYTES) holds";
    default: return "unknown status";
  }
}

extern "C" int32_t mtpattn_stream_read_default_blocks(void) {
  const int sms = device_sm_count(-1);
  return sms > 0 ? 2 * sms : MTPATTN_E_DEVICE;
}

extern "C" int mtpattn_stream_read(const void* buf, size_t bytes, uint32_t* sink, int32_t blocks,
                                   void* stream) {
  if (!buf || !sink || blocks < 0 || bytes == 0 || bytes % 16 || !aligned(buf, 16) ||
      !aligned(sink, 4))
    return MTPATTN_E_ARG;
  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess) {
    cudaGetLastError();
    return MTPATTN_E_DEVICE;
  }
  if (blocks == 0) blocks = mtpattn_stream_read_default_blocks();
  if (blocks <= 0) return MTPATTN_E_DEVICE;
  if (!on_device(buf, device) || !on_device(sink, device)) return MTPATTN_E_DEVICE;
  if (launch_stream_read(buf, bytes, sink, blocks, static_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return MTPATTN_E_LAUNCH;
  return MTPATTN_OK;
}
