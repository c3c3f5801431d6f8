// Split-KV main kernel on the sm_100-family tensor cores (tcgen05, TMA, TMEM).
//
// Scheduling.  The pages' kernel runs one work-group per (segment, sequence,
// KV head) (aiter PR #5190 page, Modifications: "grid = segments x sequences x
// kv heads").  Here every (sequence b, KV head h) unit owns max_pages_per_seq
// slots of a virtual page line, and a persistent grid of one CTA per SM cuts
// that line into equal chunks of C pages, so every SM streams the same number
// of pages.  The part of a unit inside one chunk is a "piece"; it writes its
// partial output into split slot (chunk - first chunk of the unit).  C is at
// least max_pages / (S - 1), so a unit never has more than S pieces, and the
// unit's last piece marks its unused slots empty (lse = -inf).  With S = 1,
// C = max_pages: one piece per unit.
//
// Roles, precision and TMEM layout: attn_main_common.cuh; the per-role loops:
// attn_main_body.inc, shared with planned scheduling (attn_main_planned.cu).
//
// The kernel is launched as a programmatic dependent of the previous work on the stream and
// lets the split-KV reduce be scheduled as soon as it starts.
#include "attn_main_common.cuh"

#include <algorithm>
#include <atomic>
#include <mutex>

namespace mtpattn {
namespace {

using namespace sm100;
using namespace mainkern;

struct TcParams {
  CUtensorMap tmap_k;
  CUtensorMap tmap_v;
  AttnParams a;
  int64_t unit_pages;    // W >= max_pages: virtual pages per unit
  int64_t chunk_pages;   // C
  int64_t num_chunks;    // ceil(units * W / C)
  int32_t shared_tiles;  // 1: the pieces of a unit share its tiles (see the K producer)
  int32_t pieces;        // pieces per unit when shared_tiles
};

// Position in this CTA's walk: chunk k and unit u (unit = h * num_seqs + b).
struct Cursor {
  int64_t k, u;
};

__device__ __forceinline__ Cursor cursor_first(const TcParams& prm) {
  Cursor c;
  c.k = blockIdx.x;
  // With shared tiles (one chunk per CTA) the pieces of a unit are CTAs u, u + U, u + 2U, ...
  // rather than a run of neighbouring CTAs: neighbouring CTAs tend to land on the same part
  // of the GPU, and parts of it stream at measurably different rates, so every unit gets a
  // mix and the shared tiles even it out.
  if (prm.shared_tiles) c.u = c.k % (static_cast<int64_t>(prm.a.num_seqs) * prm.a.num_kv_heads);
  else c.u = c.k * prm.chunk_pages / prm.unit_pages;
  return c;
}
__device__ __forceinline__ Cursor cursor_next(const TcParams& prm, Cursor c) {
  if (prm.shared_tiles) {                  // one unit per chunk
    c.k += gridDim.x;
    c.u = c.k % (static_cast<int64_t>(prm.a.num_seqs) * prm.a.num_kv_heads);
    return c;
  }
  const int64_t V = prm.unit_pages;
  const int64_t end = min((c.k + 1) * prm.chunk_pages,
                          static_cast<int64_t>(prm.a.num_seqs) * prm.a.num_kv_heads * V);
  ++c.u;
  if (c.u * V >= end) {
    c.k += gridDim.x;
    c.u = c.k * prm.chunk_pages / V;
  }
  return c;
}

// Geometry of one piece, computed identically by every role.
struct Item {
  int s, b, h, L, q0, ql, R, pb, pe, ntiles, err;
  int vp0;     // first virtual page of the piece (known before any load)
  int pieces;  // shared tiles: pieces of the unit
  bool last;   // the unit's last piece: it also marks the unit's unused slots empty
};

__device__ __forceinline__ Item item_info(const TcParams& prm, const Cursor& c, int lane) {
  const AttnParams& p = prm.a;
  Item x;
  x.pieces = prm.pieces;
  const int64_t V = prm.unit_pages, C = prm.chunk_pages;
  const int64_t k_first = c.u * V / C;
  if (prm.shared_tiles) {                  // slot = chunk / units; every slot of the unit runs
    x.s = static_cast<int>(c.k / (static_cast<int64_t>(p.num_seqs) * p.num_kv_heads));
    x.last = x.s == prm.pieces - 1;        // it also marks the unit's unused slots empty
  } else {
    x.s = static_cast<int>(c.k - k_first);
    x.last = c.k == (c.u * V + V - 1) / C;
  }
  x.b = static_cast<int>(c.u % p.num_seqs);
  x.h = static_cast<int>(c.u / p.num_seqs);
  const int64_t vp0 = max(c.k * C, c.u * V) - c.u * V;         // virtual page range of the piece
  const int64_t vp1 = min((c.k + 1) * C, (c.u + 1) * V) - c.u * V;
  x.vp0 = static_cast<int>(vp0);
  x.L = p.seq_lens[x.b];
  x.q0 = p.cu_q[x.b];
  const int q1 = p.cu_q[x.b + 1];
  x.ql = q1 - x.q0;
  const bool rows_known = x.q0 >= 0 && q1 <= p.total_q && x.ql >= 1 && x.ql <= kMaxQLen;
  x.err = 0;
  if (!rows_known) x.err |= MTPATTN_ERR_QLEN;
  else if (x.ql > x.L) x.err |= MTPATTN_ERR_QLEN_GT_SEQ;
  const int n_pages = x.L > 0 ? (x.L + kPage - 1) / kPage : 0;
  if (!x.err && n_pages > p.max_pages) x.err |= MTPATTN_ERR_SEQ_TOO_LONG;
  x.R = rows_known ? x.ql * p.ratio : 0;
  x.pb = x.pe = 0;
  if (!x.err) {
    x.pb = static_cast<int>(vp0);
    x.pe = static_cast<int>(min(vp1, static_cast<int64_t>(n_pages)));
    if (x.pe < x.pb) x.pe = x.pb;
  }
  if (prm.shared_tiles && !x.err) {        // the piece may take any tile of the unit
    x.pb = 0;
    x.pe = n_pages;
  }
  x.ntiles = x.err ? 0 : (x.pe - x.pb + kPagesPerTile - 1) / kPagesPerTile;
  return x;
}


// Split slots are row-major: the S slots of output row rho at rho * S .. rho * S + S - 1.
__device__ __forceinline__ float* lse_slot(const AttnParams& p, const Item& x, int r) {
  return p.lse_part + out_row(p, x, r) * p.num_segments + x.s;
}
__device__ __forceinline__ float* o_slot(const AttnParams& p, const Item& x, int r) {
  return p.o_part + (out_row(p, x, r) * p.num_segments + x.s) * kHeadDim;
}
// The unit's last piece marks the slots after its own empty.
__device__ __forceinline__ void close_unit_rows(const AttnParams& p, const Item& y, int r) {
  if (y.last)
    for (int s2 = y.s + 1; s2 < p.num_segments; ++s2)
      p.lse_part[out_row(p, y, r) * p.num_segments + s2] = -INFINITY;
}

// The CTA's first piece follows from its index alone.
__device__ __forceinline__ Cursor first_cursor_of(const TcParams& prm, Bars&, int, int,
                                                  volatile int*) {
  return cursor_first(prm);
}

// The epilogue reads the partial output from TMEM one 64-column block per round trip (two
// would not fit this kernel's registers).
constexpr int kEpilogueBlocks = 1;

__global__ void __launch_bounds__(kThreads, 1)
attn_main_tc_kernel(const __grid_constant__ TcParams prm) {
#include "attn_main_body.inc"
}

// ---- host side --------------------------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  }
  return fn;
}

// Cache view [num_pages][16][H_kv][256] bytes as a 4-D tensor (d, head, slot, page); one box is
// 128 bytes of d for one head, all 16 slots of one page, stored 128B-swizzled.
bool make_cache_map(CUtensorMap* map, const void* cache, int64_t num_pages, int hkv) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[4] = {256, static_cast<cuuint64_t>(hkv), 16, static_cast<cuuint64_t>(num_pages)};
  const cuuint64_t strides[3] = {256, static_cast<cuuint64_t>(hkv) * 256,
                                 static_cast<cuuint64_t>(hkv) * 256 * 16};
  const cuuint32_t box[4] = {128, 1, 16, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(cache), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Encoding a tensor map costs a few microseconds of host time: keep the last few.
struct MapCacheEntry {
  const void* k;
  const void* v;
  int64_t num_pages;
  int hkv;
  int device;
  CUtensorMap mk, mv;
};
std::mutex g_map_mutex;
MapCacheEntry g_map_cache[8];
int g_map_next = 0;

bool cache_maps(const AttnParams& p, int device, CUtensorMap* mk, CUtensorMap* mv) {
  std::lock_guard<std::mutex> lock(g_map_mutex);
  for (const MapCacheEntry& e : g_map_cache) {
    if (e.k == p.k_cache && e.v == p.v_cache && e.num_pages == p.num_pages &&
        e.hkv == p.num_kv_heads && e.device == device && e.k) {
      *mk = e.mk;
      *mv = e.mv;
      return true;
    }
  }
  MapCacheEntry& e = g_map_cache[g_map_next];
  if (!make_cache_map(&e.mk, p.k_cache, p.num_pages, p.num_kv_heads) ||
      !make_cache_map(&e.mv, p.v_cache, p.num_pages, p.num_kv_heads)) {
    e.k = nullptr;
    return false;
  }
  e.k = p.k_cache;
  e.v = p.v_cache;
  e.num_pages = p.num_pages;
  e.hkv = p.num_kv_heads;
  e.device = device;
  g_map_next = (g_map_next + 1) % 8;
  *mk = e.mk;
  *mv = e.mv;
  return true;
}

}  // namespace

bool kv_tensor_maps(const AttnParams& p, int device, CUtensorMap* mk, CUtensorMap* mv) {
  return cache_maps(p, device, mk, mv);
}

cudaError_t launch_attn_main(AttnParams& p, cudaStream_t stream) {
  if (p.scheduling == MTPATTN_SCHED_PLANNED) {
    const int sms = device_sm_count(-1);
    const int64_t units = static_cast<int64_t>(p.num_seqs) * p.num_kv_heads;
    if (sms > 0 && units <= kPlanUnits && units <= sms) return launch_attn_main_planned(p, stream);
  }
  p.slot_pool = 0;                         // chunked pieces keep the row-major slots
  TcParams prm;
  prm.a = p;
  if (p.num_pages > (int64_t(1) << 31) - 1) return cudaErrorInvalidValue;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!cache_maps(p, dev, &prm.tmap_k, &prm.tmap_v)) return cudaErrorInvalidValue;
  const int sms0 = device_sm_count(-1);
  if (sms0 <= 0) return cudaErrorInvalidDevice;
  const int64_t V = p.max_pages;
  const int64_t U = static_cast<int64_t>(p.num_seqs) * p.num_kv_heads;
  const int64_t S = p.num_segments;
  // Equal shares of the whole virtual page line ...
  int64_t W = V, C = V;
  if (S > 1) {
    C = (U * V + sms0 - 1) / sms0;
    const int64_t c_min = (V + S - 2) / (S - 1);
    if (C < c_min) C = c_min;
    // ... or, when every unit can get n >= 2 whole pieces for little extra per SM,
    // cut each unit into exactly n pieces (unit stride n * C) so that no chunk holds
    // two units (each extra piece costs a Q load and an epilogue on its SM).
    const int64_t n = std::min<int64_t>(sms0 / U, S);
    if (n >= 2) {
      const int64_t c_al = (V + n - 1) / n;
      if (c_al <= C + C / 8 + 16) {
        C = c_al;
        W = n * c_al;
      }
    }
  }
  prm.unit_pages = W;
  prm.chunk_pages = C;
  prm.num_chunks = (U * W + C - 1) / C;
  // When chunks never straddle units and every CTA holds one chunk, all pieces of a unit run
  // at once and may share its tiles dynamically (per-unit counters in the workspace header).
  prm.shared_tiles = (!p.deterministic && W % C == 0 && prm.num_chunks <= sms0 &&
                      U <= kMaxTileCounters) ? 1 : 0;
  prm.pieces = static_cast<int32_t>(W / C);
  // A unit of W virtual pages touches at most ceil(W / C) + 1 chunks (exactly W / C when
  // units are chunk-aligned): the reduce reads no slot beyond that.
  {
    const int64_t touch = (W % C == 0) ? W / C : (W + C - 1) / C + 1;
    p.slots_used = static_cast<int32_t>(std::min<int64_t>(touch, p.num_segments));
  }
  prm.a = p;
  static std::atomic<bool> attr_set[64];   // per device; setting it twice is harmless
  if (!attr_set[dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(attn_main_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev].store(true, std::memory_order_release);
  }
  const int grid = static_cast<int>(prm.num_chunks < sms0 ? prm.num_chunks : sms0);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, attn_main_tc_kernel, prm);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace mtpattn

#ifdef MTPATTN_TEST_COVERAGE
// Test builds only: copy the first n page counters of this kernel to host memory, then clear
// them (0 or a CUDA error code; -1 for a bad n).
extern "C" int mtpattn_test_coverage_chunked(uint32_t* host_dst, int64_t n) {
  using namespace mtpattn::mainkern;
  if (n < 0 || n > kCoverageCounters) return -1;
  void* dev = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&dev, g_coverage);
  if (e == cudaSuccess) e = cudaMemcpy(host_dst, dev, n * sizeof(uint32_t), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(dev, 0, n * sizeof(uint32_t));
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  return static_cast<int>(e);
}
#endif
