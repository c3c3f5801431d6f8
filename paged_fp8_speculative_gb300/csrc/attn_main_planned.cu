// Split-KV main kernel with planned scheduling (tcgen05, TMA, TMEM on the sm_100 family).
//
// The roles, the hi/lo e4m3 precision scheme, the TMEM layout and the online softmax are
// those of the chunked kernel in attn_main_tc.cu, and so are its per-role loops; this file
// differs in how pieces are laid out and in how a CTA finds its piece.  The two kernels are
// compiled from separate files: with both ways of scheduling in one source (a template over
// the scheduling) the hot loops ran measurably slower, a few percent at 16 x 35k tokens.
//
// Scheduling.  The chunked kernel cuts every (sequence, KV head) unit as if it held
// max_pages pages, which leaves SMs idle on ragged batches.  Here the kernel first reads
// seq_lens (plan_load / plan_piece, by the K producer warp of every CTA, all reaching the same
// result): unit v has n_v pages; the chunk C is the smallest number of pages >= one tile with
// sum_v ceil(n_v / C) <= grid and ceil(n_v / C) <= S, so the longest sequences get the most
// CTAs; unit v gets ceil(n_v / C) pieces, one per CTA, taken slot-major (slot 0 of every unit,
// then slot 1, ...) so that every unit is spread over the whole GPU.  The pieces of a unit share
// its tiles through the per-unit counter (as in the chunked kernel), or keep fixed page ranges
// [s C, (s + 1) C) in deterministic mode; the unit's last piece marks its unused slots empty.
//
// The kernel is launched as a programmatic dependent of the previous work on the stream and
// lets the split-KV reduce be scheduled as soon as it starts.
#include "common.cuh"
#include "sm100.cuh"

#include <cuda_fp8.h>
#include <math.h>

#include <algorithm>

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
  int64_t num_chunks;    // CTAs in the grid (one piece each at most)
  int32_t shared_tiles;  // 1: the pieces of a unit share its tiles (see the K producer)
  // Planned scheduling, computed on the host: per = min(S, grid / units); the chunk and the
  // pieces per unit when every unit has max_pages pages; reciprocals for exact small divisions.
  int32_t g_per, g_C, g_pu;
  float inv_units, inv_seqs, inv_per;
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
  uint64_t plan_ready;              // the CTA's piece is in plan_* (written by the K producer)
  int64_t plan_k, plan_u;
  int32_t plan_s, plan_pu, plan_C, plan_b, plan_h, plan_L, plan_q0, plan_q1;
};
static_assert(sizeof(Bars) <= 512, "barrier block");

// Position in this CTA's walk: chunk k and unit u (unit = h * num_seqs + b).
struct Cursor {
  int64_t k, u;
  int s, pu, C;            // planned scheduling: slot, pieces of the unit, pages per piece
  int b, h;                // planned scheduling: the unit's sequence and KV head
  int L, q0, q1;           // planned scheduling: the unit's seq_lens and cu_seqlens_q entries
};

// Planned scheduling (at most kPlanUnits units, no more units than CTAs): the K producer warp
// of every CTA computes the same plan from the sequence lengths.  Unit v has n_v pages; the
// chunk is the smallest C >= 8 (one tile) with sum_v ceil(n_v / C) <= grid and
// ceil(n_v / C) <= S, so the longest sequences get the most CTAs; unit v has
// p_v = ceil(n_v / C) pieces.  CTAs take the pieces slot-major (slot 0 of every unit, then
// slot 1, ...), which spreads every unit over the whole grid: neighbouring CTAs tend to share a
// part of the GPU, and parts stream at different rates.
//
// ceil(n / c) for 0 <= n < 2^24, 1 <= c, with inv = 1 / c: a float estimate, then made exact.
__device__ __forceinline__ int ceil_div_inv(int n, int c, float inv) {
  int q = __float2int_rd(static_cast<float>(n + c - 1) * inv);
  const int r = n + c - 1 - q * c;
  if (r >= c) ++q;
  if (r < 0) --q;
  return q;
}

// floor(n / d) for 0 <= n < 2^22, 1 <= d, with inv = 1 / d.
__device__ __forceinline__ int div_inv(int n, int d, float inv) {
  int q = __float2int_rz(static_cast<float>(n) * inv);
  const int r = n - q * d;
  if (r >= d) ++q;
  if (r < 0) --q;
  return q;
}

// The plan's inputs: lane l holds units l, l + 32, ... (seq_lens and the cu_seqlens_q pair of
// each).  plan_load only issues the loads, so that other requests can go out while they fly.
struct PlanIn {
  int Lv[8], q0v[8], q1v[8];
};

__device__ __forceinline__ void plan_load(const TcParams& prm, int lane, PlanIn& in) {
  const AttnParams& p = prm.a;
  const int B = p.num_seqs, U = B * p.num_kv_heads;
  const int nb = (U + 31) / 32;              // lane slots in use (warp-uniform)
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    in.Lv[i] = in.q0v[i] = in.q1v[i] = 0;
    const int v = lane + 32 * i;
    if (i < nb && v < U) {
      const int b = v - div_inv(v, B, prm.inv_seqs) * B;
      in.Lv[i] = p.seq_lens[b];
      in.q0v[i] = p.cu_q[b];                  // loaded with the lengths: item_info needs them
      in.q1v[i] = p.cu_q[b + 1];
    }
  }
}

__device__ Cursor plan_piece(const TcParams& prm, int lane, const PlanIn& in) {
  const AttnParams& p = prm.a;
  const int B = p.num_seqs, U = B * p.num_kv_heads, G = gridDim.x, S = p.num_segments;
  const int nb = (U + 31) / 32;              // lane slots in use (warp-uniform)
  const int* Lv = in.Lv;
  const int* q0v = in.q0v;
  const int* q1v = in.q1v;
  int n[8];                                  // pages of each unit
  int maxn = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    n[i] = 0;
    const int v = lane + 32 * i;
    if (i < nb && v < U) {
      const int L = Lv[i];
      const int np = L > 0 ? min((L + kPage - 1) / kPage, p.max_pages) : 0;
      n[i] = max(np, 1);                      // an empty or invalid unit still owns one piece
      maxn = max(maxn, n[i]);
    }
  }
  int minn = 0x7fffffff;                     // lanes without a unit do not count
#pragma unroll
  for (int i = 0; i < 8; ++i)
    if (i < nb && n[i] > 0) minn = min(minn, n[i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    maxn = max(maxn, __shfl_xor_sync(0xffffffffu, maxn, o));
    minn = min(minn, __shfl_xor_sync(0xffffffffu, minn, o));
  }
  if (minn == maxn) {
    // Equal lengths: the search below gives C = max(ceil(n / min(S, G / U)), one tile) and
    // ceil(n / C) pieces for every unit, which CTA k takes as slot k / U of unit k % U.  For
    // n = max_pages (the usual case) the host has worked these out.
    int C = prm.g_C, pu = prm.g_pu;
    if (maxn != p.max_pages) {
      C = max(ceil_div_inv(maxn, prm.g_per, prm.inv_per), min(kPagesPerTile, maxn));
      pu = ceil_div_inv(maxn, C, 1.f / static_cast<float>(C));
    }
    Cursor c;
    c.C = C;
    c.pu = pu;
    const int k = blockIdx.x;
    c.L = c.q0 = c.q1 = 0;
    c.b = c.h = 0;
    if (k >= U * pu) {
      c.k = prm.num_chunks;
      c.u = 0;
      c.s = 0;
    } else {
      const int ks = div_inv(k, U, prm.inv_units), ku = k - ks * U;
      c.k = k;
      c.u = ku;
      c.s = ks;
      c.h = div_inv(ku, B, prm.inv_seqs);
      c.b = ku - c.h * B;
      const int src = ku & 31, slot = ku >> 5;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int L = __shfl_sync(0xffffffffu, Lv[i], src);
        const int a = __shfl_sync(0xffffffffu, q0v[i], src);
        const int b = __shfl_sync(0xffffffffu, q1v[i], src);
        if (i == slot) {
          c.L = L;
          c.q0 = a;
          c.q1 = b;
        }
      }
    }
    return c;
  }
  int total = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) total += n[i];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) total += __shfl_xor_sync(0xffffffffu, total, o);
  auto pieces_total = [&](int c) -> int {    // sum_v ceil(n_v / c)
    const float inv = 1.f / static_cast<float>(c);
    int t = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (i < nb && n[i] > 0) t += ceil_div_inv(n[i], c, inv);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    return t;
  };
  // Bounds: sum_v ceil(n_v / c) >= total / c, and <= total / c + U, so the answer lies in
  // [ceil(total / G), ceil(total / (G - U))]; no piece is cut below one 128-key tile, and a
  // unit gets at most S pieces.
  const int hi0 = max(maxn, 1);
  int lo = max(max((total + G - 1) / G, (maxn + S - 1) / S), min(kPagesPerTile, hi0));
  int hi = G > U ? min(hi0, (total + (G - U) - 1) / (G - U)) : hi0;
  if (lo > hi0) lo = hi0;
  if (hi < lo) hi = lo;
  while (lo < hi) {
    const int mid = (lo + hi) / 2;
    if (pieces_total(mid) <= G) hi = mid;
    else lo = mid + 1;
  }
  const int C = lo;
  const float invC = 1.f / static_cast<float>(C);
  int pu[8];
  int maxp = 0, npieces = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    pu[i] = (i < nb && n[i] > 0) ? ceil_div_inv(n[i], C, invC) : 0;
    maxp = max(maxp, pu[i]);
    npieces += pu[i];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    maxp = max(maxp, __shfl_xor_sync(0xffffffffu, maxp, o));
    npieces += __shfl_xor_sync(0xffffffffu, npieces, o);
  }
  auto before = [&](int sl) -> int {         // pieces of slots below sl: sum_v min(p_v, sl)
    int t = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (i < nb) t += min(pu[i], sl);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    return t;
  };
  Cursor c;
  c.C = C;
  c.s = 0;
  c.pu = 0;
  c.u = 0;
  c.b = c.h = 0;
  const int k = blockIdx.x;
  if (k >= npieces) {                        // more CTAs than pieces: nothing for this one
    c.k = prm.num_chunks;
    return c;
  }
  int slo = 0, shi = maxp - 1;               // largest slot sl with before(sl) <= k
  while (slo < shi) {
    const int mid = (slo + shi + 1) / 2;
    if (before(mid) <= k) slo = mid;
    else shi = mid - 1;
  }
  int r = k - before(slo);                   // the r-th unit (in order) that has slot slo
  int u = -1, pu_u = 0;
  c.L = c.q0 = c.q1 = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if (i < nb) {
      const uint32_t m = __ballot_sync(0xffffffffu, pu[i] > slo);
      const int cnt = __popc(m);
      if (u < 0 && r < cnt) {
        uint32_t mm = m;
        for (int q = 0; q < r; ++q) mm &= mm - 1;        // drop the r lowest set bits
        const int ln = __ffs(mm) - 1;
        u = ln + 32 * i;
        pu_u = __shfl_sync(0xffffffffu, pu[i], ln);
        c.L = __shfl_sync(0xffffffffu, Lv[i], ln);
        c.q0 = __shfl_sync(0xffffffffu, q0v[i], ln);
        c.q1 = __shfl_sync(0xffffffffu, q1v[i], ln);
      } else if (u < 0) {
        r -= cnt;
      }
    }
  }
  c.k = k;
  c.u = u;
  c.s = slo;
  c.pu = pu_u;
  c.h = div_inv(u, B, prm.inv_seqs);
  c.b = u - c.h * B;
  return c;
}

// One piece per CTA: after it the CTA is done.
__device__ __forceinline__ Cursor cursor_next(const TcParams& prm, Cursor c) {
  c.k = prm.num_chunks;
  return c;
}

// Geometry of one piece, computed identically by every role.
struct Item {
  int s, b, h, L, q0, ql, R, pb, pe, ntiles, err;
  int vp0;     // first page of the piece's first tile (known before any load)
  int pieces;  // planned scheduling: pieces of the unit
  bool last;   // the unit's last piece: it also marks the unit's unused slots empty
};

__device__ __forceinline__ Item item_info(const TcParams& prm, const Cursor& c, int lane) {
  const AttnParams& p = prm.a;
  Item x;
  x.pieces = c.pu;                         // everything comes with the plan
  x.s = c.s;
  x.last = c.s == c.pu - 1;
  x.b = c.b;
  x.h = c.h;
  x.L = c.L;
  x.q0 = c.q0;
  const int q1 = c.q1;
  x.ql = q1 - x.q0;
  const bool rows_known = x.q0 >= 0 && q1 <= p.total_q && x.ql >= 1 && x.ql <= kMaxQLen;
  x.err = 0;
  if (!rows_known) x.err |= MTPATTN_ERR_QLEN;
  else if (x.ql > x.L) x.err |= MTPATTN_ERR_QLEN_GT_SEQ;
  const int n_pages = x.L > 0 ? (x.L + kPage - 1) / kPage : 0;
  if (!x.err && n_pages > p.max_pages) x.err |= MTPATTN_ERR_SEQ_TOO_LONG;
  x.R = rows_known ? x.ql * p.ratio : 0;
  x.pb = x.pe = 0;
  x.vp0 = prm.shared_tiles ? x.s * kPagesPerTile : x.s * c.C;
  if (!x.err) {
    if (prm.shared_tiles) {                // the piece may take any tile of the unit
      x.pb = 0;
      x.pe = n_pages;
    } else {                               // pages [s C, (s + 1) C) of the unit
      x.pb = min(x.s * c.C, n_pages);
      x.pe = min(x.pb + c.C, n_pages);
    }
  }
  x.ntiles = x.err ? 0 : (x.pe - x.pb + kPagesPerTile - 1) / kPagesPerTile;
  (void)lane;
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
attn_main_planned_kernel(const __grid_constant__ TcParams prm) {
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
    mbar_init(smem_u32(&bars.plan_ready), 1);
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

  // The CTA's piece.  The K producer warp plans and publishes the plan; the other warps take
  // it from shared memory.
  auto first_cursor = [&]() -> Cursor {
    Cursor c;
    if (warp == 0) {
      PlanIn in;
      plan_load(prm, lane, in);
      c = plan_piece(prm, lane, in);
      if (lane == 0) {
        bars.plan_k = c.k;
        bars.plan_u = c.u;
        bars.plan_s = c.s;
        bars.plan_pu = c.pu;
        bars.plan_C = c.C;
        bars.plan_b = c.b;
        bars.plan_h = c.h;
        bars.plan_L = c.L;
        bars.plan_q0 = c.q0;
        bars.plan_q1 = c.q1;
        mbar_arrive(smem_u32(&bars.plan_ready));
      }
      __syncwarp();
      return c;
    }
    const bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars.plan_ready), 0, abort_flag));
    c.k = ok ? bars.plan_k : prm.num_chunks;
    c.u = bars.plan_u;
    c.s = bars.plan_s;
    c.pu = bars.plan_pu;
    c.C = bars.plan_C;
    c.b = bars.plan_b;
    c.h = bars.plan_h;
    c.L = bars.plan_L;
    c.q0 = bars.plan_q0;
    c.q1 = bars.plan_q1;
    return c;
  };

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
    for (Cursor cur = first_cursor(); cur.k < prm.num_chunks && !stop && !*abort_flag; cur = cursor_next(prm, cur)) {
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
      //  - fixed ranges (deterministic mode): tiles 0 .. ntiles-1 of the piece (first page
      //    pb + 8 j);
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
              idx = x.s + j * x.pieces;
              if (j == 0) c0 = atomicAdd(ctr, 1u); else c1 = atomicAdd(ctr, 1u);
            } else {
              idx = 2 * x.pieces + static_cast<int>(c0);
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
        // plan alone (not from a claim), so its entries load while the first claims fly.
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
    for (Cursor cur = first_cursor(); cur.k < prm.num_chunks && !*abort_flag; cur = cursor_next(prm, cur)) {
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
    Cursor it = next_running(first_cursor(), x);
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

}  // namespace

cudaError_t launch_attn_main_planned(AttnParams& p, cudaStream_t stream) {
  TcParams prm{};
  if (p.num_pages > (int64_t(1) << 31) - 1) return cudaErrorInvalidValue;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!kv_tensor_maps(p, dev, &prm.tmap_k, &prm.tmap_v)) return cudaErrorInvalidValue;
  const int sms0 = device_sm_count(-1);
  if (sms0 <= 0) return cudaErrorInvalidDevice;
  const int64_t V = p.max_pages;
  const int64_t U = static_cast<int64_t>(p.num_seqs) * p.num_kv_heads;
  const int64_t S = p.num_segments;
  if (U > kPlanUnits || U > sms0) return cudaErrorInvalidValue;
  // One piece per CTA, at most S per unit; the pieces of a unit share its tiles unless
  // deterministic scheduling was asked for.
  prm.shared_tiles = p.deterministic ? 0 : 1;
  prm.num_chunks = std::min<int64_t>(sms0, U * S);
  // With equal lengths every unit gets min(S, grid / U) pieces: the reduce reads that many
  // slots with the LSEs and the others only if a unit used them.
  const int64_t per = std::min<int64_t>(S, prm.num_chunks / U);
  p.slots_used = static_cast<int32_t>(per);
  // The plan of equal lengths (every unit max_pages pages), the plan's fast path; reciprocals
  // for exact small divisions on the device.
  const int64_t Cg = std::max<int64_t>((V + per - 1) / per, std::min<int64_t>(kPagesPerTile, V));
  prm.g_per = static_cast<int32_t>(per);
  prm.g_C = static_cast<int32_t>(Cg);
  prm.g_pu = static_cast<int32_t>((V + Cg - 1) / Cg);
  prm.inv_units = 1.f / static_cast<float>(U);
  prm.inv_seqs = 1.f / static_cast<float>(p.num_seqs);
  prm.inv_per = 1.f / static_cast<float>(per);
  prm.a = p;
  static bool attr_set[64] = {false};
  if (!attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(attn_main_planned_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(prm.num_chunks));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, attn_main_planned_kernel, prm);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace mtpattn
