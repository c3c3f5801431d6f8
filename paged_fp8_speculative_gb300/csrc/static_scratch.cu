// mtp_verify_attn_fwd_static_scratch: the same operation as mtp_verify_attn_fwd
// for callers that cannot allocate device memory.
//
// Some callers have no way to obtain a workspace: a plain C host that runs
// inside another framework's memory pool and may not call cudaMalloc, code
// that issues its launches while a CUDA graph is being captured (where a fresh
// cudaMalloc is not allowed), or a latency-critical loop that must never hit
// cudaMalloc / cudaFree because they can synchronise the device.  For them the
// split-KV partials live in one file-scope device array that the library owns
// for the life of the process, MTPATTN_STATIC_SCRATCH_BYTES on every GPU that
// loads the library.
//
// The array's host-side name is only a stand-in for the symbol, not a device
// address, so the address the kernels get comes from cudaGetSymbolAddress,
// looked up once per device with that device current (on the first call on
// that device) and cached.  Every call shares the array: calls that overlap on
// the GPU race on it.
//
// The workspace's counter header (its first kWorkspaceHeaderBytes) must be zero
// before the first call; every call that runs both of its kernels leaves its tile
// counters zero and its two call counters equal, and the partials behind it need
// no clearing.  The header is cleared
// with cudaMemsetAsync on the caller's stream, so the clear is ordered before
// the call's kernels whatever kind of stream the caller uses: on the first call
// on each device, and on the next call after one whose reduce could not be
// launched (E_LAUNCH), which may have left the counters non-zero.
#include "common.cuh"

#include <mutex>

namespace {

static __device__ __align__(256) unsigned char g_static_scratch[MTPATTN_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {nullptr};
bool g_header_dirty[kMaxDevices] = {false};   // the header must be cleared before the next call

// Device address of the scratch array on `device` (the current device), with its header
// cleared on `stream` if that is still owed (nullptr on failure).  Called under the mutex.
void* scratch_address(int device, cudaStream_t stream) {
  if (device < 0 || device >= kMaxDevices) return nullptr;
  if (!g_scratch_addr[device]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || !ptr) {
      cudaGetLastError();
      return nullptr;
    }
    g_scratch_addr[device] = ptr;
    g_header_dirty[device] = true;          // the entry state: clear once, in stream order
  }
  if (g_header_dirty[device]) {
    if (cudaMemsetAsync(g_scratch_addr[device], 0, mtpattn::kWorkspaceHeaderBytes, stream) !=
        cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    g_header_dirty[device] = false;
  }
  return g_scratch_addr[device];
}

}  // namespace

extern "C" int mtp_verify_attn_fwd_static_scratch(
    const void* q, int64_t q_stride_tok, int64_t q_stride_head, const void* k_cache,
    const void* v_cache, int64_t num_pages, const int32_t* block_tables,
    int32_t max_pages_per_seq, const int32_t* seq_lens, const int32_t* cu_seqlens_q,
    int32_t num_seqs, int32_t total_q, int32_t num_q_heads, int32_t num_kv_heads,
    const float* k_descale, const float* v_descale, float softmax_scale, int32_t num_segments,
    void* out, int64_t out_stride_tok, int64_t out_stride_head, int32_t* status, void* stream) {
  if (num_seqs == 0 && total_q == 0) return MTPATTN_OK;
  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess) {
    cudaGetLastError();
    return MTPATTN_E_DEVICE;
  }
  // 0 stays 0 in the call below (the library then chooses S, and may share the slots out by
  // length); the size check uses the S it will choose.
  int32_t s_resolved = num_segments;
  if (num_segments == 0 && num_seqs > 0 && num_kv_heads > 0 && max_pages_per_seq > 0) {
    s_resolved = mtp_verify_attn_num_segments(num_seqs, num_kv_heads, max_pages_per_seq, device);
    if (s_resolved < 1) return MTPATTN_E_DEVICE;
  }
  const size_t need = mtp_verify_attn_workspace_size(total_q, num_q_heads, s_resolved);
  if (need > static_cast<size_t>(MTPATTN_STATIC_SCRATCH_BYTES)) return MTPATTN_E_SCRATCH_LIMIT;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  void* scratch = scratch_address(device, st);
  if (!scratch) return MTPATTN_E_DEVICE;
  const int rc = mtp_verify_attn_fwd(q, q_stride_tok, q_stride_head, k_cache, v_cache, num_pages,
                                     block_tables, max_pages_per_seq, seq_lens, cu_seqlens_q,
                                     num_seqs, total_q, num_q_heads, num_kv_heads, k_descale,
                                     v_descale, softmax_scale, num_segments, scratch,
                                     static_cast<size_t>(MTPATTN_STATIC_SCRATCH_BYTES), out,
                                     out_stride_tok, out_stride_head, status, stream);
  // A failed launch may come after the main kernel ran without the reduce that resets the
  // tile counters: clear the header again before the next call.
  if (rc == MTPATTN_E_LAUNCH) g_header_dirty[device] = true;
  return rc;
}
