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
// Roles (352 threads):
//   warp 0     K producer: per piece, first the piece's bf16 query rows (plain bulk copies
//              into the Q buffer), then TMA loads of its K pages straight from the paged NHD
//              cache through the block table (two 128-byte-wide boxes per page, 128B-swizzled)
//              into a 3-stage ring;
//   warp 10    V producer: the same for V (a V slot frees one tile later than a K slot);
//   warp 1     MMA warp: runs warp-uniformly, one elected lane issues the tcgen05.mma
//              instructions and their commits; it owns the TMEM allocation;
//   warps 2-9  softmax: warp (quadrant q = w & 3, half g) owns TMEM lanes 32q + 16g .. +15.
//
// Precision.  Both contractions run as e4m3 x e4m3 -> f32 MMAs on the cache bytes
// themselves, so K and V are never converted.  Q and P keep bf16-class precision by writing
// each as the sum of two e4m3 terms:
//   Q:  x = q * 2^a (a per row, so max|x| is in [128, 256)),
//       hi = e4m3(x), lo = e4m3((x - hi) * 16);  x = hi + lo/16 exactly for every element
//       within 2^-13 of the row maximum (a bf16 value has 8 significant bits: hi keeps 4
//       and the remainder fits lo's 4);
//   P:  p_s = 2^(s - m + 8 - kTau) in [0, 256] as hi + lo/16 the same way.
// The hi and lo rows are stacked into one M = 128 MMA: query row r = 16q + 8g + a has its
// hi row in TMEM lane 32q + 16g + a and its lo row 8 lanes below.  With the 16x256b access
// shape one thread holds both lanes of its row, so S = hi + lo/16 is formed in registers,
// and O = O_hi + O_lo/16 likewise in the epilogue.
//
// Online softmax with a lazy reference: m is only raised (and O rescaled in TMEM) when a
// tile's row maximum exceeds it by more than kTau (log2 units); otherwise p <= 2^kTau,
// which the P encoding scale 2^(8 - kTau) absorbs.
//
// Tile = 128 keys (8 pages).  TMEM: S double buffer at columns 0 and 128 (the tile's P
// overwrites the first 32 columns of its S buffer, 4 e4m3 per column), O at columns
// 256..511.  QK is 8 MMAs (K = 32 bytes each) with A = stacked Q and B = the K tile (both
// K-major); PV is 4 MMAs with A = P from TMEM and B = the V tile read MN-major.  The MMA
// warp issues QK(u), PV(u-1), QK(u+1), ...: QK(u + 2) reuses the S buffer whose P(u) PV(u)
// reads, and needs no wait for it because the MMAs of one thread execute in issue order.
//
// The kernel is launched as a programmatic dependent of the previous work on the stream and
// lets the split-KV reduce be scheduled as soon as it starts.
#include "common.cuh"
#include "sm100.cuh"

#include <cuda_fp8.h>
#include <math.h>

#include <algorithm>
#include <mutex>

namespace mtpattn {
namespace {

using namespace sm100;

constexpr int kThreads = 352;
constexpr int kSoftmaxThreads = 256;
constexpr int kTileKeys = 128;
constexpr int kPagesPerTile = kTileKeys / kPage;       // 8
constexpr int kHalfBytes = kTileKeys * 128;            // one 128-byte column half of a tile
constexpr int kTileBytes = 2 * kHalfBytes;             // 32 KB per tensor per tile
constexpr int kStages = 3;
constexpr int kQBytes = 128 * 256;                     // stacked hi/lo Q, two halves of 16 KB
constexpr int kSCols = 128;
constexpr int kOCol = 256;
constexpr int kTmemCols = 512;
constexpr float kTau = 3.f;                            // lazy-rescale threshold (log2 units)
constexpr float kPShift = 8.f - kTau;                  // p_s = p * 2^kPShift <= 256

// Shared-memory map (offsets from a 1024-byte-aligned base).  The whole 227 KB
// is requested; the kernel checks that the aligned layout fits before using it.
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kQBytes;
constexpr int kOffV = kOffK + kStages * kTileBytes;
constexpr int kOffBar = kOffV + kStages * kTileBytes;
constexpr int kOffXchg = kOffBar + 512;                // 2 x 2 x 128 floats of cross-group exchange
constexpr int kLayoutBytes = kOffXchg + 2 * 2 * 128 * 4;
constexpr int kSmemBytes = 232448;
static_assert(kLayoutBytes + 512 <= kSmemBytes, "shared-memory layout");

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

constexpr int kRing = 16;              // entries of the tile-sequence ring

struct Bars {
  uint64_t k_full[kStages], k_empty[kStages], v_full[kStages], v_empty[kStages];
  uint64_t s_full[2], p_full[2], pv_done[2];
  uint64_t q_ready, final_mma;
  uint64_t q_land;                  // the piece's bf16 Q rows have landed in the Q buffer
  uint64_t q_free;                  // the piece's last QK has completed: the Q buffer may be refilled
  uint64_t xbar[2];                 // cross-group exchange, one per slot parity
  uint64_t tid_full[kRing];         // ring entry e written (arrival count 1: the K producer)
  int32_t tid[kRing];               // first page of the piece's next tile, or -1: piece done
  uint32_t tmem_base;
  int32_t abort;
};
static_assert(sizeof(Bars) <= 512, "barrier block");

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
  bool last;   // the unit's last piece: it also marks the unit's unused slots empty
};

__device__ __forceinline__ Item item_info(const TcParams& prm, const Cursor& c, int lane) {
  const AttnParams& p = prm.a;
  Item x;
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


__device__ __forceinline__ int64_t out_row(const AttnParams& p, const Item& x, int r) {
  const int t = r / p.ratio, g = r - t * p.ratio;
  return static_cast<int64_t>(x.q0 + t) * p.num_q_heads + x.h * p.ratio + g;
}

// Split x0..x3 into hi codes (4 bytes) and lo codes (4 bytes): x = hi + lo / 16.
// hi = e4m3(x); the remainder x - hi is formed in f16 (exact: x rounded to f16 keeps 11
// significant bits, hi 4, and their difference fits), scaled by 16 and rounded to e4m3.
__device__ __forceinline__ void split4(float x0, float x1, float x2, float x3, uint32_t& hi,
                                       uint32_t& lo) {
  asm("{\n"
      " .reg .b16 h01, h23, l01, l23;\n"
      " .reg .b32 x01, x23, g01, g23, r01, r23, s16;\n"
      " cvt.rn.satfinite.e4m3x2.f32 h01, %3, %2;\n"
      " cvt.rn.satfinite.e4m3x2.f32 h23, %5, %4;\n"
      " cvt.rn.f16x2.f32 x01, %3, %2;\n"
      " cvt.rn.f16x2.f32 x23, %5, %4;\n"
      " cvt.rn.f16x2.e4m3x2 g01, h01;\n"
      " cvt.rn.f16x2.e4m3x2 g23, h23;\n"
      " mov.b32 s16, 0x4C004C00;\n"
      " sub.rn.f16x2 r01, x01, g01;\n"
      " sub.rn.f16x2 r23, x23, g23;\n"
      " mul.rn.f16x2 r01, r01, s16;\n"
      " mul.rn.f16x2 r23, r23, s16;\n"
      " cvt.rn.satfinite.e4m3x2.f16x2 l01, r01;\n"
      " cvt.rn.satfinite.e4m3x2.f16x2 l23, r23;\n"
      " mov.b32 %0, {h01, h23};\n"
      " mov.b32 %1, {l01, l23};\n"
      "}\n"
      : "=r"(hi), "=r"(lo)
      : "f"(x0), "f"(x1), "f"(x2), "f"(x3));
}

__device__ __forceinline__ float pow2f(int e) {  // 2^e for e in [-126, 127]
  return __int_as_float((e + 127) << 23);
}
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  float2 c;
  asm("{\n .reg .b64 ra, rb, rc;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mul.rn.f32x2 rc, ra, rb;\n mov.b64 {%0, %1}, rc;\n}\n"
      : "=f"(c.x), "=f"(c.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return c;
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  float2 c;
  asm("{\n .reg .b64 ra, rb, rc;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " add.rn.f32x2 rc, ra, rb;\n mov.b64 {%0, %1}, rc;\n}\n"
      : "=f"(c.x), "=f"(c.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return c;
}
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {  // a * b + c
  float2 d;
  asm("{\n .reg .b64 ra, rb, rc, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mov.b64 rc, {%6, %7};\n fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;\n}\n"
      : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float ex2(float x) {  // 2^x, hardware approximation (rel. err ~2^-22)
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

__global__ void __launch_bounds__(kThreads, 1)
attn_main_tc_kernel(const __grid_constant__ TcParams prm) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  if (base + kLayoutBytes > smem_raw + kSmemBytes) {     // uniform across the CTA
    if (threadIdx.x == 0) set_status(prm.a.status, MTPATTN_ERR_TIMEOUT);
    return;
  }
  Bars& bars = *reinterpret_cast<Bars*>(base + kOffBar);
  float* xchg = reinterpret_cast<float*>(base + kOffXchg);   // [parity][group][128 lanes]
  const AttnParams& p = prm.a;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int* abort_flag = &bars.abort;

  // ---- set-up ------------------------------------------------------------------------------
  if (warp == 1) {
    tmem_alloc(smem_u32(&bars.tmem_base), kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(smem_u32(&bars.k_full[i]), 1);
      mbar_init(smem_u32(&bars.k_empty[i]), 1);
      mbar_init(smem_u32(&bars.v_full[i]), 1);
      mbar_init(smem_u32(&bars.v_empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bars.s_full[i]), 1);
      mbar_init(smem_u32(&bars.p_full[i]), kSoftmaxThreads);
      mbar_init(smem_u32(&bars.pv_done[i]), 1);
    }
    mbar_init(smem_u32(&bars.q_ready), kSoftmaxThreads);
    mbar_init(smem_u32(&bars.final_mma), 1);
    mbar_init(smem_u32(&bars.q_land), 1);
    mbar_init(smem_u32(&bars.q_free), 1);
    mbar_init(smem_u32(&bars.xbar[0]), kSoftmaxThreads);
    mbar_init(smem_u32(&bars.xbar[1]), kSoftmaxThreads);
    for (int i = 0; i < kRing; ++i) mbar_init(smem_u32(&bars.tid_full[i]), 1);
    bars.abort = 0;
    fence_mbar_init();
  }
  // The V ring must hold finite values before any P = 0 column meets it.
  for (int i = tid; i < (kStages * kTileBytes) / 16; i += kThreads)
    reinterpret_cast<uint4*>(base + kOffV)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;
  // Launched as a programmatic dependent of the previous work on the stream: the set-up
  // above touched no global memory; from here on inputs are read and the workspace is
  // written, so wait until that work has completed and its results are visible.
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  // The segment reduce may be scheduled now; it waits for this grid's results itself.
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");

  if (warp == 0 || warp == 10) {
    // ================================ producers (K: warp 0, V: warp 10) ============================
    const bool is_v = warp == 10;
    const CUtensorMap* map = is_v ? &prm.tmap_v : &prm.tmap_k;
    uint64_t* full = is_v ? bars.v_full : bars.k_full;
    uint64_t* empty = is_v ? bars.v_empty : bars.k_empty;
    const int ring = is_v ? kOffV : kOffK;
    if (lane == 0) prefetch_tmap(map);
    const uint64_t pol = l2_policy_evict_first();
    uint32_t t = 0;    // tiles issued by this producer
    uint32_t e = 0;    // entries of the tile-sequence ring passed (tiles and end marks)
    uint32_t n_q = 0;  // pieces whose Q rows this (K) producer has copied
    bool stop = false;
    for (Cursor cur = cursor_first(prm); cur.k < prm.num_chunks && !stop && !*abort_flag; cur = cursor_next(prm, cur)) {
      const Item x = item_info(prm, cur, lane);
      if (x.ntiles == 0) continue;
      const int32_t* bt = p.block_tables + static_cast<size_t>(x.b) * p.max_pages;
      // Q rows of the piece (K producer only): row r (token r / ratio, head h * ratio +
      // r % ratio) to byte r * 512 of the Q buffer, once the previous piece's last QK has
      // stopped reading that buffer.  Each copy instruction costs the TMA unit tens of
      // cycles, so when the heads of a token are contiguous (the usual layout) one copy
      // moves all `ratio` rows of a token.
      auto copy_q = [&]() -> bool {
        bool q_ok = true;
        if (lane == 0) {
          q_ok = mbar_wait(smem_u32(&bars.q_free), (n_q & 1) ^ 1, abort_flag);
          if (q_ok) mbar_arrive_expect_tx(smem_u32(&bars.q_land), x.R * 2 * kHeadDim);
        }
        q_ok = __shfl_sync(0xffffffffu, q_ok, 0);
        if (!q_ok) return false;
        if (p.q_stride_head == kHeadDim) {
          if (lane < x.ql)
            bulk_load(smem_u32(base + kOffQ + lane * p.ratio * 2 * kHeadDim),
                      p.q + static_cast<int64_t>(x.q0 + lane) * p.q_stride_tok +
                          static_cast<int64_t>(x.h) * p.ratio * kHeadDim,
                      p.ratio * 2 * kHeadDim, smem_u32(&bars.q_land));
        } else {
          for (int r = lane; r < x.R; r += 32) {
            const int tk = r / p.ratio, g = r - tk * p.ratio;
            const __nv_bfloat16* src = p.q + static_cast<int64_t>(x.q0 + tk) * p.q_stride_tok +
                                       static_cast<int64_t>(x.h * p.ratio + g) * p.q_stride_head;
            bulk_load(smem_u32(base + kOffQ + r * 2 * kHeadDim), src, 2 * kHeadDim,
                      smem_u32(&bars.q_land));
          }
        }
        ++n_q;
        return true;
      };
      // The piece's tile sequence is decided by the K producer and handed to every other
      // role through the ring (first page of each tile, then -1).
      //  - chunks: tiles 0 .. ntiles-1 of the piece (first page pb + 8 j);
      //  - shared tiles (each CTA holds one piece, all pieces of a unit run together): piece s
      //    of n takes tiles s and s + n of the unit, then tiles 2n + c with c claimed from the
      //    unit's counter, so the unit's CTAs finish within about a tile of each other
      //    whatever bandwidth each SM gets.  Claims run two tiles ahead of their use, and a
      //    thread's successive claims increase, so a claim past the end is never followed by
      //    a valid one it would drop.
      uint32_t* ctr = p.tile_ctr + cur.u;
      uint32_t c0 = 0, c1 = 0;                 // lane 0: claims in flight
      for (int j = 0; ; ++j) {
        int pg0 = -1;
        if (!is_v) {
          int idx = -1;
          if (lane == 0) {
            if (!prm.shared_tiles) {
              idx = j < x.ntiles ? j : -1;
            } else if (j < 2) {
              idx = x.s + j * prm.pieces;
              if (j == 0) c0 = atomicAdd(ctr, 1u); else c1 = atomicAdd(ctr, 1u);
            } else {
              idx = 2 * prm.pieces + static_cast<int>(c0);
              c0 = c1;
              if (idx < x.ntiles) c1 = atomicAdd(ctr, 1u);
            }
            if (idx >= x.ntiles) idx = -1;
          }
          idx = __shfl_sync(0xffffffffu, idx, 0);
          pg0 = idx < 0 ? -1 : x.pb + idx * kPagesPerTile;
        } else {
          const bool got = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars.tid_full[e % kRing]),
                                                             (e / kRing) & 1, abort_flag));
          if (!got) {
            stop = true;
            break;
          }
          pg0 = bars.tid[e % kRing];
        }
        if (pg0 < 0) {                         // end of the piece's sequence
          if (!is_v && lane == 0) {
            bars.tid[e % kRing] = -1;
            mbar_arrive(smem_u32(&bars.tid_full[e % kRing]));
          }
          ++e;
          if (j == 0 && !is_v && !copy_q()) stop = true;   // an empty piece still gets its Q
          break;
        }
        const int np = min(kPagesPerTile, x.pe - pg0);
        const int st = t % kStages;
        // One page per lane, loads in parallel.  The first tile's address comes from the
        // cursor alone, so its entries are fetched together with the piece's lengths.
        const int pg_first = prm.shared_tiles ? x.s * kPagesPerTile : x.vp0;
        const int pg_spec = (j == 0 ? pg_first : pg0) + lane;
        int phys = (lane < kPagesPerTile && pg_spec < p.max_pages) ? bt[pg_spec] : 0;
        if (lane >= np) phys = 0;
        const uint32_t fb = smem_u32(&full[st]);
        bool ok = true;
        if (lane == 0) {
          // Start-up: the first K tile goes out ahead of the other K tiles (and of every V
          // tile), so that it is not queued behind them.
          if ((t == 1 && !is_v) || (t == 0 && is_v))
            ok = mbar_wait(smem_u32(&bars.k_full[0]), 0, abort_flag);
          ok = ok && mbar_wait(smem_u32(&empty[st]), ((t / kStages) & 1) ^ 1, abort_flag);
          if (ok) {
            if (!is_v) {                       // published once its K slot is free (ring bound)
              bars.tid[e % kRing] = pg0;
              mbar_arrive(smem_u32(&bars.tid_full[e % kRing]));
            }
            mbar_arrive_expect_tx(fb, np * 2 * 2048);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
          stop = true;
          break;
        }
        if (lane < np) {
          const uint32_t dst = smem_u32(base + ring + st * kTileBytes);
          tma_load_4d(dst + lane * 2048, map, fb, 0, x.h, 0, phys, pol);
          tma_load_4d(dst + kHalfBytes + lane * 2048, map, fb, 128, x.h, 0, phys, pol);
        }
        ++t;
        ++e;
        // The piece's first K tile is on the way; its Q rows follow.
        if (j == 0 && !is_v && !copy_q()) {
          stop = true;
          break;
        }
      }
    }
    // Never leave with copies in flight: wait for the last Q rows and the last issued tiles.
    if (lane == 0 && n_q > 0) {
      volatile int no_abort = 0;
      mbar_wait(smem_u32(&bars.q_land), (n_q - 1) & 1, &no_abort);
    }
    if (lane == 0) {
      for (uint32_t k = 0; k < kStages && k < t; ++k) {
        const uint32_t u = t - 1 - k;
        volatile int no_abort = 0;
        mbar_wait(smem_u32(&full[u % kStages]), (u / kStages) & 1, &no_abort);
      }
    }
  } else if (warp == 1) {
    // ======================================= MMA issuer =========================================
    // The whole warp runs the loop, so every value it uses is warp-uniform; one elected lane
    // issues the MMAs and their commits (a commit tracks the MMAs of the lane that issues it).
    // The shared-memory descriptors are built once: operands move by whole 16-byte units,
    // so advancing the 14-bit start-address field by (offset >> 4) never carries out of it.
    constexpr uint32_t kIdescQK = idesc_e4m3_f32(128, kTileKeys, false);
    constexpr uint32_t kIdescPV = idesc_e4m3_f32(128, kHeadDim, true);
    const uint64_t q_desc = sdesc_sw128(smem_u32(base + kOffQ), 16, 1024);
    const uint64_t k_desc = sdesc_sw128(smem_u32(base + kOffK), 16, 1024);
    const uint64_t v_desc = sdesc_sw128(smem_u32(base + kOffV), kHalfBytes, 1024);
    const bool leader = elect_one();
    uint32_t t = 0;
    uint32_t items_run = 0;
    auto wait_all = [&](uint64_t& bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(smem_u32(&bar), parity, abort_flag));
    };
    auto issue_pv = [&](uint32_t u, bool first) -> bool {
      const int st = u % kStages;
      if (!wait_all(bars.v_full[st], (u / kStages) & 1)) return false;
      if (!wait_all(bars.p_full[u & 1], (u >> 1) & 1)) return false;
      tc_fence_after();
      if (leader) {
        const uint32_t p_tmem = tmem + (u & 1) * kSCols;
#pragma unroll
        for (int k = 0; k < kTileKeys / 32; ++k)
          mma_f8_ts(tmem + kOCol, p_tmem + 8 * k, v_desc + ((st * kTileBytes + k * 4096) >> 4),
                    kIdescPV, (first && k == 0) ? 0u : 1u);
        mma_commit(smem_u32(&bars.v_empty[st]));
        mma_commit(smem_u32(&bars.pv_done[u & 1]));
      }
      __syncwarp();
      return true;
    };
    uint32_t e = 0;                            // tile-sequence ring entries passed
    for (Cursor cur = cursor_first(prm); cur.k < prm.num_chunks && !*abort_flag; cur = cursor_next(prm, cur)) {
      const Item x = item_info(prm, cur, lane);
      if (x.ntiles == 0) continue;
      bool ok = wait_all(bars.q_ready, items_run & 1);
      tc_fence_after();
      int j = 0;                               // tiles of this piece
      while (ok) {
        if (!wait_all(bars.tid_full[e % kRing], (e / kRing) & 1)) { ok = false; break; }
        const int pg0 = bars.tid[e % kRing];
        ++e;
        if (pg0 < 0) break;
        const uint32_t u = t;
        const int st = u % kStages;
        // S buffer u & 1 still holds P(u - 2) for PV(u - 2).  That PV was issued before this
        // QK by this warp, and MMAs of one thread execute in issue order, so it reads P(u - 2)
        // before QK(u) overwrites it: no wait on its completion is needed.
        if (!wait_all(bars.k_full[st], (u / kStages) & 1)) { ok = false; break; }
        tc_fence_after();
        if (leader) {
#pragma unroll
          for (int k = 0; k < kHeadDim / 32; ++k) {
            const uint32_t a_off = (k >> 2) * (kQBytes / 2) + (k & 3) * 32;
            const uint32_t b_off = st * kTileBytes + (k >> 2) * kHalfBytes + (k & 3) * 32;
            mma_f8_ss(tmem + (u & 1) * kSCols, q_desc + (a_off >> 4), k_desc + (b_off >> 4),
                      kIdescQK, k > 0 ? 1u : 0u);
          }
          mma_commit(smem_u32(&bars.s_full[u & 1]));
          mma_commit(smem_u32(&bars.k_empty[st]));
        }
        __syncwarp();
        if (j > 0 && !issue_pv(u - 1, j == 1)) { ok = false; break; }
        ++t;
        ++j;
      }
      if (!ok) break;
      // Every QK of the piece is issued: the Q buffer is free once they complete.
      if (leader) mma_commit(smem_u32(&bars.q_free));
      __syncwarp();
      if (j > 0 && !issue_pv(t - 1, j == 1)) break;
      ++items_run;
    }
    if (leader) mma_commit(smem_u32(&bars.final_mma));
    __syncwarp();
    {
      volatile int no_abort = 0;
      mbar_wait(smem_u32(&bars.final_mma), 0, &no_abort);
    }
  } else {
    // ======================================= softmax warps =======================================
    // Warp (quadrant q, half g) owns TMEM lanes 32q + 16g .. +15: query rows r = 16q + 8g + a
    // (a < 8), hi in lane 32q + 16g + a and lo 8 lanes below.  With the 16x256b access shape
    // thread t holds both lanes of row a = t/4 for the column pairs 8j + 2(t%4) (+1), so the
    // hi + lo/16 sum is local and a row max takes two shuffles.
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;
    const int c4 = lane & 3;
    const int arow = lane >> 2;
    const int rloc = 16 * quad + 8 * half + arow;           // query row of this thread
    const uint32_t blk_addr = tmem + (static_cast<uint32_t>(32 * quad + 16 * half) << 16);
    // Q preparation writes A row 32q + lane, half `half` of its 256 bytes.
    const int L32 = 32 * quad + lane;
    const bool q_is_hi = (lane & 15) < 8;
    const int q_row = 16 * quad + 8 * (lane >> 4) + (lane & 7);
    const float kd = __ldg(p.k_descale);
    const float vd = __ldg(p.v_descale);
    const bool even = (c4 & 1) == 0;                         // even: writes P_hi of the row
    const uint32_t sel_lo = even ? 0x5410u : 0x1054u;        // byte selectors of the P words
    const uint32_t sel_hi = even ? 0x7632u : 0x3276u;

    // The unit's unused split slots (after its last piece) are empty: lse = -inf, and the
    // reduce never reads the partial output of a slot whose weight is 0.
    auto close_unit = [&](const Item& y) {
      if (y.last && c4 == 0 && rloc < y.R)
        for (int s2 = y.s + 1; s2 < p.num_segments; ++s2)
          p.lse_part[out_row(p, y, rloc) * p.num_segments + s2] = -INFINITY;
    };
    // Pieces with nothing to compute: an error gets a NaN LSE (the reduce writes zeros),
    // an empty piece an empty slot.
    auto trivial_item = [&](const Item& y) {
      if (c4 == 0 && rloc < y.R)
        p.lse_part[out_row(p, y, rloc) * p.num_segments + y.s] =
            y.err ? __int_as_float(0x7fc00000) : -INFINITY;
      if (y.err && lane == 0 && warp == 2) set_status(p.status, y.err);
      close_unit(y);
    };
    // First piece with tiles at or after cursor c (finishing trivial pieces on the way).
    auto next_running = [&](Cursor c, Item& y) -> Cursor {
      for (; c.k < prm.num_chunks; c = cursor_next(prm, c)) {
        y = item_info(prm, c, lane);
        if (y.ntiles > 0) return c;
        trivial_item(y);
      }
      return c;
    };
    // Value exchange with the same lane of warp (quad, half ^ 1) through shared memory and
    // the xbar barriers (all 256 softmax threads arrive; the barrier alternates per call).
    int xpar = 0;
    uint32_t xphase = 0;
    auto exchange = [&](float v, float& other) -> bool {
      xchg[(xpar * 2 + half) * 128 + L32] = v;
      mbar_arrive(smem_u32(&bars.xbar[xpar]));
      const bool ok = __all_sync(0xffffffffu,
                                 mbar_wait(smem_u32(&bars.xbar[xpar]), (xphase >> xpar) & 1, abort_flag));
      other = xchg[(xpar * 2 + (half ^ 1)) * 128 + L32];
      xphase ^= 1u << xpar;
      xpar ^= 1;
      return ok;
    };
    // Q of piece y into the stacked A tile.  The producer has bulk-copied the piece's bf16
    // rows into the Q buffer (row r at byte r * 512).  The pair of lanes l (hi A row of query
    // row q_row) and l ^ 8 (its lo A row) shares that row's half `half`: each reads 64 of its
    // 128 values and writes their hi codes to the hi A row and lo codes to the lo A row.  The
    // row's scale 2^a (max |q| * 2^a in [128, 256)) needs the max over both halves, which
    // sit in warp (quad, half ^ 1): the exchange gives it, and since every thread arrives
    // only after its reads, it also frees the buffer for the codes that overwrite it.
    uint32_t q_par = 0;
    auto prepare_q = [&](const Item& y, int& a_exp_row) -> bool {
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars.q_land), q_par, abort_flag))) return false;
      q_par ^= 1;
      int a_exp = 0;
      const bool valid = q_row < y.R;
      const int part = q_is_hi ? 0 : 1;
      uint4 w[8];                                // chunk (i + lane) & 7: no bank conflicts
      float mx = 0.f;
      if (valid) {
        const unsigned char* src = base + kOffQ + q_row * 2 * kHeadDim + half * kHeadDim + part * 128;
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i] = *reinterpret_cast<const uint4*>(src + ((i + lane) & 7) * 16);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint32_t ww[4] = {w[i].x, w[i].y, w[i].z, w[i].w};
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(ww[k] << 16)),
                                 fabsf(__uint_as_float(ww[k] & 0xFFFF0000u))));
        }
      }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
      float mx_other;
      if (!exchange(mx, mx_other)) return false;
      mx = fmaxf(mx, mx_other);
      if (mx > 0.f) {
        int e;
        frexpf(mx, &e);                          // mx = f * 2^e, f in [0.5, 1)
        a_exp = min(126, max(-126, 8 - e));      // mx * 2^a in [128, 256)
      }
      const float sc = pow2f(a_exp);
      const int l_hi = 32 * quad + (lane & ~8);
      unsigned char* row_hi = base + kOffQ + half * (kQBytes / 2) + l_hi * 128;
      unsigned char* row_lo = row_hi + 8 * 128;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int c = (i + lane) & 7;            // source chunk: codes 8c .. 8c + 7 of this part
        uint2 hi = make_uint2(0u, 0u), lo = make_uint2(0u, 0u);
        if (valid) {
          const uint32_t a0 = w[i].x, a1 = w[i].y, a2 = w[i].z, a3 = w[i].w;
          split4(__uint_as_float(a0 << 16) * sc, __uint_as_float(a0 & 0xFFFF0000u) * sc,
                 __uint_as_float(a1 << 16) * sc, __uint_as_float(a1 & 0xFFFF0000u) * sc, hi.x, lo.x);
          split4(__uint_as_float(a2 << 16) * sc, __uint_as_float(a2 & 0xFFFF0000u) * sc,
                 __uint_as_float(a3 << 16) * sc, __uint_as_float(a3 & 0xFFFF0000u) * sc, hi.y, lo.y);
        }
        const int byte = part * 64 + c * 8;      // within the 128-byte half row, before swizzling
        const int off = (((byte >> 4) ^ (l_hi & 7)) << 4) + (byte & 15);
        *reinterpret_cast<uint2*>(row_hi + off) = hi;
        *reinterpret_cast<uint2*>(row_lo + off) = lo;
      }
      fence_proxy_async_smem();
      mbar_arrive(smem_u32(&bars.q_ready));
      // this thread's softmax row (rloc) is A rows 32q+16g+a / +8: lane 16g + a of this warp
      a_exp_row = __shfl_sync(0xffffffffu, a_exp, 16 * half + arow);
      return true;
    };

    uint32_t t = 0;                            // tiles processed
    uint32_t e = 0;                            // tile-sequence ring entries passed
    Item x;
    Cursor it = next_running(cursor_first(prm), x);
    int a_exp = 0;
    bool alive = it.k >= prm.num_chunks || prepare_q(x, a_exp);
    while (alive && it.k < prm.num_chunks) {
      const bool row_valid = rloc < x.R;
      const bool warp_active = __any_sync(0xffffffffu, row_valid);
      const int tk = row_valid ? rloc / p.ratio : 0;
      // last visible key of this row, clipped to the piece's pages
      const int vis_max = row_valid ? min(x.L - x.ql + tk, x.pe * kPage - 1) : -1;
      const float sscale = p.scale_log2 * kd * pow2f(-a_exp);
      const float2 w_hi = make_float2(sscale, sscale);
      const float2 w_lo = make_float2(sscale * 0.0625f, sscale * 0.0625f);
      float m_ref = -INFINITY, l_part = 0.f;
      Item xn;                                 // next piece
      Cursor itn;
      itn.k = prm.num_chunks;
      itn.u = 0;
      int a_next = 0;
      // Whether a block-table entry of the piece lies outside the page pool: each tile's
      // entries (read by the producers just before, so from L1) are checked during the tile.
      bool bad = false;
      const int32_t* bt_row = p.block_tables + static_cast<size_t>(x.b) * p.max_pages;

      int j = 0;                               // tiles of this piece
      for (;; ++j) {
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars.tid_full[e % kRing]), (e / kRing) & 1, abort_flag))) { alive = false; break; }
        const int pg0 = bars.tid[e % kRing];   // first page of the tile, or -1: piece done
        ++e;
        if (pg0 < 0) break;
        const uint32_t u = t + j;
        const uint32_t sb = u & 1;
        const int pg_lane = pg0 + lane;
        const int32_t bt_e = (lane < kPagesPerTile && pg_lane < x.pe) ? bt_row[pg_lane] : 0;
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars.s_full[sb]), (u >> 1) & 1, abort_flag))) { alive = false; break; }
        tc_fence_after();
        float s[32];                           // s[2jj + e]: key 8jj + 2 c4 + e of the tile
        float alpha = 1.f;
        bool rescale = false;
        uint32_t pw[16];
        if (warp_active) {
          uint32_t v0[32], v1[32];
          tmem_ld16x256_x8(blk_addr + sb * kSCols, v0);
          tmem_ld16x256_x8(blk_addr + sb * kSCols + 64, v1);
          tmem_ld_wait(v0);
          tmem_ld_wait(v1);
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            const float2 h0 = make_float2(__uint_as_float(v0[4 * jj]), __uint_as_float(v0[4 * jj + 1]));
            const float2 l0 = make_float2(__uint_as_float(v0[4 * jj + 2]), __uint_as_float(v0[4 * jj + 3]));
            const float2 h1 = make_float2(__uint_as_float(v1[4 * jj]), __uint_as_float(v1[4 * jj + 1]));
            const float2 l1 = make_float2(__uint_as_float(v1[4 * jj + 2]), __uint_as_float(v1[4 * jj + 3]));
            const float2 c0 = ffma2(l0, w_lo, fmul2(h0, w_hi));
            const float2 c1 = ffma2(l1, w_lo, fmul2(h1, w_hi));
            s[2 * jj] = c0.x; s[2 * jj + 1] = c0.y;
            s[16 + 2 * jj] = c1.x; s[17 + 2 * jj] = c1.y;
          }
          const int key0 = pg0 * kPage + 2 * c4;
          if (!__all_sync(0xffffffffu, key0 - 2 * c4 + kTileKeys - 1 <= vis_max)) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (key0 + 8 * (i >> 1) + (i & 1) > vis_max) s[i] = -INFINITY;
          }
          float m8[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) m8[i] = fmaxf(fmaxf(s[i], s[i + 8]), fmaxf(s[i + 16], s[i + 24]));
#pragma unroll
          for (int i = 0; i < 4; ++i) m8[i] = fmaxf(m8[i], m8[i + 4]);
          float mx = fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3]));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
          // lazy reference: raise m only when the tile beats it by more than kTau
          if (mx != -INFINITY && (m_ref == -INFINITY || mx > m_ref + kTau)) {
            if (m_ref != -INFINITY) {
              alpha = ex2(m_ref - mx);
              rescale = true;
            }
            m_ref = mx;
          }
          const float2 moff = make_float2(kPShift - m_ref, kPShift - m_ref);  // p_s = 2^(s - m + shift)
          uint32_t hiw[8], low[8];
          float2 ps2 = make_float2(0.f, 0.f);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            // s[2k], s[2k+1]: keys of column pair jj = k (first 64 keys) ... packed per split4 as
            // (jj = 2m, 2m+1) so each word's halves are two consecutive pairs.
            const int i0 = (k < 4) ? 4 * k : 16 + 4 * (k - 4);
            const float2 e01 = fadd2(make_float2(s[i0], s[i0 + 1]), moff);
            const float2 e23 = fadd2(make_float2(s[i0 + 2], s[i0 + 3]), moff);
            const float2 p01 = make_float2(ex2(e01.x), ex2(e01.y));   // s = -inf gives 0
            const float2 p23 = make_float2(ex2(e23.x), ex2(e23.y));
            ps2 = fadd2(ps2, fadd2(p01, p23));
            split4(p01.x, p01.y, p23.x, p23.y, hiw[k], low[k]);
          }
          l_part = l_part * alpha + (ps2.x + ps2.y);
          // P words: word of pair jj (keys 8jj + 4(c4>>1) .. +3) is built by the even/odd thread
          // pair c4, c4^1: even keeps its hi bytes and takes the partner's, odd likewise for lo.
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t own = even ? hiw[k] : low[k];
            const uint32_t snd = even ? low[k] : hiw[k];
            const uint32_t rcv = __shfl_xor_sync(0xffffffffu, snd, 1);
            pw[2 * k] = __byte_perm(own, rcv, sel_lo);
            pw[2 * k + 1] = __byte_perm(own, rcv, sel_hi);
          }
          // P goes to its S buffer's first 32 columns (it does not depend on O).
          tmem_st16x64_x16(blk_addr + sb * kSCols, pw);
        }
        // O may only be touched once the previous tile's PV has completed
        if (j > 0) {
          if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars.pv_done[(u - 1) & 1]), ((u - 1) >> 1) & 1, abort_flag))) { alive = false; break; }
          tc_fence_after();
          if (warp_active && __any_sync(0xffffffffu, rescale)) {
            const float2 a2 = make_float2(alpha, alpha);
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
              uint32_t a0[32];
              tmem_ld16x256_x8(blk_addr + kOCol + 64 * c, a0);
              tmem_ld_wait(a0);
#pragma unroll
              for (int i = 0; i < 32; i += 2) {
                const float2 r0 = fmul2(make_float2(__uint_as_float(a0[i]), __uint_as_float(a0[i + 1])), a2);
                a0[i] = __float_as_uint(r0.x);
                a0[i + 1] = __float_as_uint(r0.y);
              }
              tmem_st16x256_x8(blk_addr + kOCol + 64 * c, a0);
            }
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(smem_u32(&bars.p_full[sb]));
        bad |= __any_sync(0xffffffffu, bt_e < 0 || bt_e >= p.num_pages);
      }
      // All QK of this piece are complete (s_full of its last tile was waited), so Q can be
      // rewritten for the next piece while this piece's last PV runs.
      if (alive && !__any_sync(0xffffffffu, *abort_flag != 0)) {
        itn = cursor_next(prm, it);
        if (itn.k < prm.num_chunks) xn = item_info(prm, itn, lane);
        if (itn.k < prm.num_chunks && xn.ntiles == 0) {
          trivial_item(xn);
          itn = next_running(cursor_next(prm, itn), xn);
        }
        if (itn.k < prm.num_chunks && !prepare_q(xn, a_next)) alive = false;
      }
      if (!alive || __any_sync(0xffffffffu, *abort_flag != 0)) break;

      // ---- epilogue: o = v_descale * (O_hi + O_lo / 16) / l, lse = m + log2 l -----------------
      // (a piece may have taken no tile of its unit: then nothing was accumulated, lse = -inf)
      if (j > 0) {
        const uint32_t ul = t + j - 1;
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars.pv_done[ul & 1]), (ul >> 1) & 1, abort_flag))) break;
        tc_fence_after();
      }
      float l = l_part + __shfl_xor_sync(0xffffffffu, l_part, 1);
      l += __shfl_xor_sync(0xffffffffu, l, 2);   // sum of p_s over the row's visible keys
      if (warp_active) {
        const float oscale = l > 0.f ? vd / l : 0.f;
        const float2 wh = make_float2(oscale, oscale);
        const float2 wl = make_float2(oscale * 0.0625f, oscale * 0.0625f);
        float* orow = row_valid ? p.o_part + (out_row(p, x, rloc) * p.num_segments + x.s) * kHeadDim : nullptr;
#pragma unroll 1
        for (int c = 0; c < (j > 0 ? 4 : 0); ++c) {
          uint32_t a0[32];
          tmem_ld16x256_x8(blk_addr + kOCol + 64 * c, a0);
          tmem_ld_wait(a0);
          if (row_valid) {
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
              const float2 h = make_float2(__uint_as_float(a0[4 * jj]), __uint_as_float(a0[4 * jj + 1]));
              const float2 lo = make_float2(__uint_as_float(a0[4 * jj + 2]), __uint_as_float(a0[4 * jj + 3]));
              const float2 o = ffma2(lo, wl, fmul2(h, wh));
              *reinterpret_cast<float2*>(orow + 64 * c + 8 * jj + 2 * c4) = o;
            }
          }
        }
        if (c4 == 0 && row_valid)
          p.lse_part[out_row(p, x, rloc) * p.num_segments + x.s] =
              bad ? __int_as_float(0x7fc00000) : (l > 0.f ? m_ref + log2f(l) - kPShift : -INFINITY);
        if (bad && lane == 0) set_status(p.status, MTPATTN_ERR_PAGE);
      }
      close_unit(x);
      tc_fence_before();
      t += j;
      x = xn;
      it = itn;
      a_exp = a_next;
    }
  }

  // ---- teardown ------------------------------------------------------------------------------
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (*abort_flag && tid == 0) set_status(p.status, MTPATTN_ERR_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
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
  static bool attr_set[64] = {false};
  if (!attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(attn_main_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
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
