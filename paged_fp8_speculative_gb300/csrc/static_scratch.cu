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
// the GPU race on it.  The workspace's counter header must be zero when a call
// starts: the array is cleared once, on the first call on its device, and every
// call leaves the header zero again (the partials need no clearing).
#include "common.cuh"

#include <mutex>

namespace {

static __device__ __align__(256) unsigned char g_static_scratch[MTPATTN_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device (nullptr on failure).
void* scratch_address(int device) {
  if (device < 0 || device >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_addr[device]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || !ptr ||
        cudaMemset(ptr, 0, MTPATTN_STATIC_SCRATCH_BYTES) != cudaSuccess) {   // the entry state
      cudaGetLastError();
      return nullptr;
    }
    g_scratch_addr[device] = ptr;
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
  if (num_segments == 0 && num_seqs > 0 && num_kv_heads > 0 && max_pages_per_seq > 0) {
    num_segments = mtp_verify_attn_num_segments(num_seqs, num_kv_heads, max_pages_per_seq, device);
    if (num_segments < 1) return MTPATTN_E_DEVICE;
  }
  const size_t need = mtp_verify_attn_workspace_size(total_q, num_q_heads, num_segments);
  if (need > static_cast<size_t>(MTPATTN_STATIC_SCRATCH_BYTES)) return MTPATTN_E_SCRATCH_LIMIT;
  void* scratch = scratch_address(device);
  if (!scratch) return MTPATTN_E_DEVICE;
  return mtp_verify_attn_fwd(q, q_stride_tok, q_stride_head, k_cache, v_cache, num_pages,
                             block_tables, max_pages_per_seq, seq_lens, cu_seqlens_q, num_seqs,
                             total_q, num_q_heads, num_kv_heads, k_descale, v_descale,
                             softmax_scale, num_segments, scratch,
                             static_cast<size_t>(MTPATTN_STATIC_SCRATCH_BYTES), out,
                             out_stride_tok, out_stride_head, status, stream);
}
