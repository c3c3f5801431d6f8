// Definitions shared by the two compilations of the split-KV main kernel (planned scheduling
// in attn_main_planned.cu, chunked scheduling in attn_main_tc.cu, both built around the body in
// attn_main_body.inc): tile and ring geometry, the shared-memory and TMEM maps, the barrier
// block, and the arithmetic helpers of the softmax warps.
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
// The fp8 Q/P tier (a second compilation of the planned kernel with MTPATTN_QP_FP8 set,
// the precision class of the pages' kernel, "Q and P are quantized to fp8") keeps the same
// layout and MMAs but writes only the hi codes: x = hi (lo rows zero) for Q, and p_s = hi
// for P, so each is one e4m3 rounding (3 mantissa bits) of the same scaled value.
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
#pragma once

#include <cuda_fp8.h>
#include <math.h>

#include "common.cuh"
#include "sm100.cuh"

namespace mtpattn {
namespace mainkern {

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
  int32_t plan_pool, plan_off;
};
static_assert(sizeof(Bars) <= 512, "barrier block");

// Output row (token-major, head-minor) of row r of piece x: token r / ratio, head h * ratio + r % ratio.
template <class ItemT>
__device__ __forceinline__ int64_t out_row(const AttnParams& p, const ItemT& x, int r) {
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

#if MTPATTN_QP_FP8
// The fp8 Q/P tier (attn_main_planned_qp8.cu): x0..x3 rounded to single e4m3 codes (lowest
// byte first, the byte order of split4's hi word), round to nearest even, saturating.
__device__ __forceinline__ uint32_t e4m3x4(float x0, float x1, float x2, float x3) {
  uint32_t r;
  asm("{\n"
      " .reg .b16 a, b;\n"
      " cvt.rn.satfinite.e4m3x2.f32 a, %2, %1;\n"
      " cvt.rn.satfinite.e4m3x2.f32 b, %4, %3;\n"
      " mov.b32 %0, {a, b};\n"
      "}\n"
      : "=r"(r)
      : "f"(x0), "f"(x1), "f"(x2), "f"(x3));
  return r;
}
#endif

#ifdef MTPATTN_TEST_COVERAGE
// Test builds only: how often each (sequence, KV head, logical page) had its K streamed, one
// counter per page of a [num_seqs][num_kv_heads][max_pages_per_seq] grid (each compilation of
// the kernel has its own array; the including file exports a reader).
constexpr int64_t kCoverageCounters = int64_t(1) << 22;
static __device__ uint32_t g_coverage[kCoverageCounters];
__device__ __forceinline__ void coverage_count(const AttnParams& p, int b, int h, int page) {
  const int64_t i = (static_cast<int64_t>(b) * p.num_kv_heads + h) * p.max_pages + page;
  if (i >= 0 && i < kCoverageCounters) atomicAdd(&g_coverage[i], 1u);
}
#endif

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

}  // namespace mainkern
}  // namespace mtpattn
