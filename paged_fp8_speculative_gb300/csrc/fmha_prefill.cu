// fp8 varlen prefill attention, query/key head dim 192 and value head dim 128, on the
// sm_100-family tensor cores (tcgen05, TMA, TMEM): the second workload of the library
// (aiter PR #7375 page, "Summary" and "Changes": e4m3 q/k/v with per-tensor descales, packed
// varlen THD layout, bf16 output, optional log-sum-exp, causal bottom-right or not).
//
// Work: one CTA per (128-query tile, query head, sequence); for a causal call the tiles of a
// head run last-to-first, so the heaviest tiles start first.  Roles (320 threads):
//   warps 0-15 softmax, four groups of four warps: warp w owns query rows 32 (w % 4) .. +31
//              (TMEM lanes; a warp may only reach the lanes of its own quarter) and group w / 4
//              owns keys 32 (w / 4) .. +31 of every 128-key tile and output dims 32 (w / 4) ..
//              +31.  The groups of a row exchange their maxima once per tile through shared
//              memory, so all take the same decisions.  The softmax is issue bound, and four
//              warps per SM sub-partition hide its latencies far better than one;
//   warp 16    TMA: the Q tile once, then K tiles (128 keys) and V tiles into 3-stage rings;
//   warp 17    MMA: one elected lane issues tcgen05.mma kind::f8f6f4 and the commits, and
//              the warp owns the TMEM allocation.
// A 192-byte q or k row is staged as two 128-byte-swizzled halves of 128 rows; the upper
// half's columns 192..255 lie past the tensor's head dim, and TMA fills them with zeros,
// but QK only runs over bytes 0..191 (6 MMAs of K = 32).  The V tile is 128 keys x 128 bytes,
// read MN-major as the B operand of PV.
//
// Precision: Q, K and V are the e4m3 inputs themselves.  P keeps bf16-class precision as
// two e4m3 terms, p = hi + lo / 16 (hi = e4m3(p), lo = e4m3(16 (p - hi))), each multiplied
// with V by its own MMA into its own accumulator: O = O_hi + O_lo / 16.  A single e4m3 P
// (4 significant bits) puts about 4% of noise on every weight, 0.2-0.3 std of error on
// long rows of comparable logits.
//
// TMEM: S double buffer at columns 0 and 128 (fp32), O_hi at 256..383, O_lo at 384..511.
// Group g writes its 32 keys' P_hi codes into columns 32 g .. 32 g + 7 of the tile's S buffer
// and P_lo into 32 g + 8 .. + 15 (4 codes per column, inside the columns it read itself), and
// PV takes A = P from TMEM.  The MMA warp
// issues QK(j), PV(j-1), QK(j+1), ...: QK(j+2) reuses the buffer whose P(j) PV(j) reads, and
// the MMAs of one thread execute in issue order.
//
// Online softmax in the log2 domain with a lazy reference m (raised, and O rescaled in TMEM,
// only when a tile's row maximum exceeds it by more than kTau): p_s = 2^(s - m + kShift)
// <= 2^8, so P fits e4m3 and a probability 2^-14 below the row's maximum is still a
// non-zero code (the probability-underflow case of the aiter PR #7375 page's review).
#include "common.cuh"
#include "sm100.cuh"

#include "../../include/fmha_fp8_varlen.h"

#include <cuda_fp8.h>
#include <math.h>

#include <mutex>

namespace mtpattn {
namespace {

using namespace sm100;

constexpr int kGroupsP = 4;                     // softmax groups of 4 warps
constexpr int kColsP = 128 / kGroupsP;          // keys (and output dims) per group
constexpr int kSoftmaxP = kGroupsP * 128;
constexpr int kThreadsP = kSoftmaxP + 64;
constexpr int kWarpTma = kSoftmaxP / 32, kWarpMma = kWarpTma + 1;
constexpr int kBM = 128;                        // query rows per tile
constexpr int kBN = 128;                        // keys per tile
constexpr int kHalfP = 128 * 128;               // one 128-byte-wide half of 128 rows (16 KB)
constexpr int kQTile = 2 * kHalfP;              // 32 KB
constexpr int kKTile = 2 * kHalfP;              // 32 KB per K stage
constexpr int kVTile = kHalfP;                  // 16 KB per V stage
constexpr int kStagesP = 3;
constexpr int kOffQP = 0;
constexpr int kOffKP = kOffQP + kQTile;
constexpr int kOffVP = kOffKP + kStagesP * kKTile;
constexpr int kOffBarP = kOffVP + kStagesP * kVTile;
constexpr int kOffXP = kOffBarP + 256;          // [2 tile parities][groups][128 rows] floats
constexpr int kLayoutP = kOffXP + 2 * kGroupsP * 128 * 4;
constexpr int kSmemP = kLayoutP + 1024;         // + alignment slack
constexpr int kTmemColsP = 512;
constexpr int kOColP = 256;                     // O_hi; O_lo at kOColP + 128
constexpr float kTau = 3.f;                     // lazy-rescale threshold (log2 units)
constexpr float kShift = 8.f - kTau;            // p_s = 2^(s - m + kShift) <= 2^8
constexpr float kLn2 = 0.6931471805599453f;

struct PrefillParams {
  CUtensorMap tmap_q, tmap_k, tmap_v;
  const int32_t* cu_q;
  const int32_t* cu_k;
  int32_t num_seqs, total_q, total_k, hq, hkv, ratio, n_qtiles, causal;
  const float* q_descale;
  const float* k_descale;
  const float* v_descale;
  float scale_log2;                             // softmax_scale * log2(e)
  __nv_bfloat16* out;
  int64_t out_stride_tok, out_stride_head;
  float* lse;                                   // optional [hq][total_q]
  int32_t* status;                              // optional
};

struct PBars {
  uint64_t q_full;
  uint64_t k_full[kStagesP], k_empty[kStagesP], v_full[kStagesP], v_empty[kStagesP];
  uint64_t s_full[2], p_full[2], pv_done[2];
  uint64_t final_mma;
  uint64_t xbar[4][2];              // row-quarter q, tile parity: the groups' exchange (4 x 32 arrivals)
  uint32_t tmem_base;
  int32_t abort;
};
static_assert(sizeof(PBars) <= 256, "barrier block");

__device__ __forceinline__ float ex2f(float x) {   // 2^x, hardware approximation
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

// The two-term e4m3 encoding of four probabilities p0..p3 (f32): hw = e4m3(p) (4 codes, lowest
// byte first) and lw = e4m3(16 (p - hi)), formed in f16x2 arithmetic: p rounded to f16 keeps
// 11 significant bits, hi decodes exactly into f16 (every e4m3 value is an f16 normal) and
// p - hi is exact in f16 (|p - hi| <= p / 16), so the pair carries p to f16's precision.
__device__ __forceinline__ void p_encode4(float p0, float p1, float p2, float p3, uint32_t& hw,
                                          uint32_t& lw) {
  asm("{\n .reg .b32 p01, p23, g01, g23, s16;\n"
      " .reg .b16 a, b, c, d;\n"
      " cvt.rn.f16x2.f32 p01, %3, %2;\n"
      " cvt.rn.f16x2.f32 p23, %5, %4;\n"
      " cvt.rn.satfinite.e4m3x2.f16x2 a, p01;\n"
      " cvt.rn.satfinite.e4m3x2.f16x2 b, p23;\n"
      " cvt.rn.f16x2.e4m3x2 g01, a;\n"
      " cvt.rn.f16x2.e4m3x2 g23, b;\n"
      " mov.b32 s16, 0x4C004C00;\n"
      " sub.rn.f16x2 g01, p01, g01;\n"
      " sub.rn.f16x2 g23, p23, g23;\n"
      " mul.rn.f16x2 g01, g01, s16;\n"
      " mul.rn.f16x2 g23, g23, s16;\n"
      " cvt.rn.satfinite.e4m3x2.f16x2 c, g01;\n"
      " cvt.rn.satfinite.e4m3x2.f16x2 d, g23;\n"
      " mov.b32 %0, {a, b};\n"
      " mov.b32 %1, {c, d};\n"
      "}\n"
      : "=r"(hw), "=r"(lw)
      : "f"(p0), "f"(p1), "f"(p2), "f"(p3));
}

__global__ void __launch_bounds__(kThreadsP, 1)
fmha_fp8_prefill_kernel(const __grid_constant__ PrefillParams prm) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- the CTA's tile (uniform across the CTA) ------------------------------------------------
  const int tix = blockIdx.x % prm.n_qtiles;
  const int rest = blockIdx.x / prm.n_qtiles;
  const int h = rest % prm.hq;
  const int b = rest / prm.hq;
  const int t = prm.causal ? prm.n_qtiles - 1 - tix : tix;
  const int q0 = prm.cu_q[b], q1 = prm.cu_q[b + 1];
  const int k0 = prm.cu_k[b], k1 = prm.cu_k[b + 1];
  const bool cu_ok = q0 >= 0 && q0 <= q1 && q1 <= prm.total_q && k0 >= 0 && k0 <= k1 &&
                     k1 <= prm.total_k && q1 - q0 <= prm.n_qtiles * kBM;
  if (!cu_ok) {
    if (tid == 0 && tix == 0 && h == 0) set_status(prm.status, FMHA_FP8_ERR_CU);
    return;
  }
  const int Lq = q1 - q0, Lk = k1 - k0, i0 = t * kBM;
  if (i0 >= Lq) return;
  // keys the tile needs: all Lk, or (causal) up to the last row's reach i + Lk - Lq
  int kneed = Lk;
  if (prm.causal) kneed = min(Lk, max(0, min(i0 + kBM, Lq) - 1 + Lk - Lq + 1));
  const int nt = (kneed + kBN - 1) / kBN;
  const int hk = h / prm.ratio;

  if (nt == 0) {                      // no visible key in the tile: zeros and lse -inf
    if (tid < kBM && i0 + tid < Lq) {
      const int64_t row = q0 + i0 + tid;
      uint4* dst = reinterpret_cast<uint4*>(prm.out + row * prm.out_stride_tok +
                                            static_cast<int64_t>(h) * prm.out_stride_head);
#pragma unroll
      for (int i = 0; i < 16; ++i) dst[i] = make_uint4(0u, 0u, 0u, 0u);
      if (prm.lse) prm.lse[static_cast<int64_t>(h) * prm.total_q + row] = -INFINITY;
    }
    return;
  }

  PBars& bars = *reinterpret_cast<PBars*>(base + kOffBarP);
  volatile int* abort_flag = &bars.abort;

  // ---- set-up -----------------------------------------------------------------------------------
  if (warp == kWarpMma) {
    tmem_alloc(smem_u32(&bars.tmem_base), kTmemColsP);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(smem_u32(&bars.q_full), 1);
    for (int i = 0; i < kStagesP; ++i) {
      mbar_init(smem_u32(&bars.k_full[i]), 1);
      mbar_init(smem_u32(&bars.k_empty[i]), 1);
      mbar_init(smem_u32(&bars.v_full[i]), 1);
      mbar_init(smem_u32(&bars.v_empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bars.s_full[i]), 1);
      mbar_init(smem_u32(&bars.p_full[i]), kSoftmaxP);
      mbar_init(smem_u32(&bars.pv_done[i]), 1);
    }
    mbar_init(smem_u32(&bars.final_mma), 1);
    for (int q = 0; q < 4; ++q)
      for (int par = 0; par < 2; ++par) mbar_init(smem_u32(&bars.xbar[q][par]), kGroupsP * 32);
    bars.abort = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;

  if (warp == kWarpTma) {
    // ===================================== TMA producer ==========================================
    if (lane == 0) {
      prefetch_tmap(&prm.tmap_q);
      prefetch_tmap(&prm.tmap_k);
      prefetch_tmap(&prm.tmap_v);
      const uint32_t qb = smem_u32(&bars.q_full);
      mbar_arrive_expect_tx(qb, kQTile);
      tma_load_3d(smem_u32(base + kOffQP), &prm.tmap_q, qb, 0, h, q0 + i0);
      tma_load_3d(smem_u32(base + kOffQP + kHalfP), &prm.tmap_q, qb, 128, h, q0 + i0);
      int j = 0;
      for (; j < nt; ++j) {
        const int st = j % kStagesP;
        const uint32_t ph = (j / kStagesP) & 1;
        if (!mbar_wait(smem_u32(&bars.k_empty[st]), ph ^ 1, abort_flag)) break;
        const uint32_t kb = smem_u32(&bars.k_full[st]);
        mbar_arrive_expect_tx(kb, kKTile);
        const uint32_t kd = smem_u32(base + kOffKP + st * kKTile);
        tma_load_3d(kd, &prm.tmap_k, kb, 0, hk, k0 + j * kBN);
        tma_load_3d(kd + kHalfP, &prm.tmap_k, kb, 128, hk, k0 + j * kBN);
        if (!mbar_wait(smem_u32(&bars.v_empty[st]), ph ^ 1, abort_flag)) {
          ++j;                           // its K copy is in flight: wait for it below
          break;
        }
        const uint32_t vb = smem_u32(&bars.v_full[st]);
        mbar_arrive_expect_tx(vb, kVTile);
        tma_load_3d(smem_u32(base + kOffVP + st * kVTile), &prm.tmap_v, vb, 0, hk, k0 + j * kBN);
      }
      // Never leave with copies in flight (only after an abort can some be unconsumed).
      volatile int no_abort = 0;
      mbar_wait(smem_u32(&bars.q_full), 0, &no_abort);
      for (int u = max(0, j - kStagesP); u < j; ++u) {
        mbar_wait(smem_u32(&bars.k_full[u % kStagesP]), (u / kStagesP) & 1, &no_abort);
        mbar_wait(smem_u32(&bars.v_full[u % kStagesP]), (u / kStagesP) & 1, &no_abort);
      }
    }
  } else if (warp == kWarpMma) {
    // ===================================== MMA issuer ============================================
    constexpr uint32_t kIdescQK = idesc_e4m3_f32(kBM, kBN, false);
    constexpr uint32_t kIdescPV = idesc_e4m3_f32(kBM, 128, true);
    const uint64_t q_desc = sdesc_sw128(smem_u32(base + kOffQP), 16, 1024);
    const uint64_t k_desc = sdesc_sw128(smem_u32(base + kOffKP), 16, 1024);
    const uint64_t v_desc = sdesc_sw128(smem_u32(base + kOffVP), kHalfP, 1024);
    const bool leader = elect_one();
    auto wait_all = [&](uint64_t& bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(smem_u32(&bar), parity, abort_flag));
    };
    auto issue_pv = [&](int u) -> bool {
      const int st = u % kStagesP;
      if (!wait_all(bars.v_full[st], (u / kStagesP) & 1)) return false;
      if (!wait_all(bars.p_full[u & 1], (u >> 1) & 1)) return false;
      tc_fence_after();
      if (leader) {
        const uint32_t p_tmem = tmem + (u & 1) * 128;
        // keys 32 k .. 32 k + 31 (group k): P_hi at column 32 k, P_lo at 32 k + 8
#pragma unroll
        for (int k = 0; k < kBN / 32; ++k)                 // O_hi += P_hi V
          mma_f8_ts(tmem + kOColP, p_tmem + 32 * k, v_desc + ((st * kVTile + k * 4096) >> 4),
                    kIdescPV, (u > 0 || k > 0) ? 1u : 0u);
#pragma unroll
        for (int k = 0; k < kBN / 32; ++k)                 // O_lo += P_lo V
          mma_f8_ts(tmem + kOColP + 128, p_tmem + 32 * k + 8,
                    v_desc + ((st * kVTile + k * 4096) >> 4), kIdescPV, (u > 0 || k > 0) ? 1u : 0u);
        mma_commit(smem_u32(&bars.v_empty[st]));
        mma_commit(smem_u32(&bars.pv_done[u & 1]));
      }
      __syncwarp();
      return true;
    };
    bool ok = wait_all(bars.q_full, 0);
    for (int j = 0; ok && j < nt; ++j) {
      const int st = j % kStagesP;
      if (!wait_all(bars.k_full[st], (j / kStagesP) & 1)) { ok = false; break; }
      tc_fence_after();
      if (leader) {
#pragma unroll
        for (int k = 0; k < 6; ++k) {                 // head-dim bytes 32k .. 32k + 31 (of 192)
          const uint32_t a_off = (k >> 2) * kHalfP + (k & 3) * 32;
          const uint32_t b_off = st * kKTile + (k >> 2) * kHalfP + (k & 3) * 32;
          mma_f8_ss(tmem + (j & 1) * 128, q_desc + (a_off >> 4), k_desc + (b_off >> 4), kIdescQK,
                    k > 0 ? 1u : 0u);
        }
        mma_commit(smem_u32(&bars.s_full[j & 1]));
        mma_commit(smem_u32(&bars.k_empty[st]));
      }
      __syncwarp();
      if (j > 0 && !issue_pv(j - 1)) ok = false;
    }
    if (ok) issue_pv(nt - 1);
    if (leader) mma_commit(smem_u32(&bars.final_mma));
    __syncwarp();
    volatile int no_abort = 0;
    mbar_wait(smem_u32(&bars.final_mma), 0, &no_abort);
  } else {
    // ===================================== softmax (rows) ========================================
    const int quad = warp & 3;                                // TMEM lane quarter
    const int grp = warp >> 2;                                // keys / dims kColsP grp .. + kColsP - 1
    const int r = 32 * quad + lane;                           // query row of the tile, TMEM lane
    const int i = i0 + r;
    const bool valid = i < Lq;
    // last key index row i may see (within the sequence)
    const int lim = !valid ? -1 : (prm.causal ? min(Lk - 1, i + Lk - Lq) : Lk - 1);
    const float sl2 = prm.scale_log2 * __ldg(prm.q_descale) * __ldg(prm.k_descale);
    const float vd = __ldg(prm.v_descale);
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * quad) << 16);
    const uint32_t col0 = kColsP * grp;                       // this group's S / P / O columns
    float* xch = reinterpret_cast<float*>(base + kOffXP);     // [parity][group][row]
    // Exchange with the same row in the other groups (warps quad + 4 g): use k of parity slot
    // par is its (k / 2)-th use; every wait is bounded, so a group that gave up (abort) cannot
    // leave the others waiting.  Returns the maximum (is_max) or the sum over the groups.
    auto exchange = [&](int use, float v, bool is_max, float& all) -> bool {
      const int par = use & 1;
      xch[(par * kGroupsP + grp) * 128 + r] = v;
      mbar_arrive(smem_u32(&bars.xbar[quad][par]));
      const bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars.xbar[quad][par]),
                                                        (use >> 1) & 1, abort_flag));
      all = xch[(par * kGroupsP) * 128 + r];
#pragma unroll
      for (int g2 = 1; g2 < kGroupsP; ++g2) {
        const float o = xch[(par * kGroupsP + g2) * 128 + r];
        all = is_max ? fmaxf(all, o) : all + o;
      }
      return ok;
    };
    float m = -INFINITY, l = 0.f;
    bool alive = true;
    for (int j = 0; j < nt; ++j) {
      const int sb = j & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars.s_full[sb]), (j >> 1) & 1, abort_flag))) {
        alive = false;
        break;
      }
      tc_fence_after();
      float s[kColsP];                                        // raw logits <q, k> (unscaled)
      {
        uint32_t v[32];
        tmem_ld32(lane_addr + sb * 128 + col0, v);
        tmem_ld_wait(v);
#pragma unroll
        for (int e = 0; e < 32; ++e) s[e] = __uint_as_float(v[e]);
      }
      const int key0 = j * kBN + col0;
      const bool masked = key0 + kColsP - 1 > lim;            // some key past the row's reach
      if (masked) {                                           // out of the maximum below
#pragma unroll
        for (int e = 0; e < kColsP; ++e)
          if (key0 + e > lim) s[e] = sl2 >= 0.f ? -INFINITY : INFINITY;
      }
      // the largest scaled logit: sl2 times the largest (sl2 >= 0) or smallest raw one
      float hm;
      if (sl2 >= 0.f) {
        float a = fmaxf(s[0], s[1]), b = fmaxf(s[2], s[3]);
#pragma unroll
        for (int e = 4; e < kColsP; e += 4) {
          a = fmaxf(a, fmaxf(s[e], s[e + 1]));
          b = fmaxf(b, fmaxf(s[e + 2], s[e + 3]));
        }
        hm = fmaxf(a, b) * sl2;
      } else {
        float a = s[0];
#pragma unroll
        for (int e = 1; e < kColsP; ++e) a = fminf(a, s[e]);
        hm = a * sl2;
      }
      if (hm != hm) hm = -INFINITY;                           // 0 * inf (sl2 = 0, masked)
      float mx;                                               // the tile's row maximum
      if (!exchange(j, hm, true, mx)) {
        alive = false;
        break;
      }
      float alpha = 1.f;
      bool rescale = false;
      if (mx != -INFINITY && (m == -INFINITY || mx > m + kTau)) {
        if (m != -INFINITY) {
          alpha = ex2f(m - mx);
          rescale = true;
        }
        m = mx;
      }
      const float moff = m == -INFINITY ? 0.f : kShift - m;   // all s are -inf while m is
      float psum;
      {
        // p = 2^(sl2 s + kShift - m); masked keys get 2^-inf = 0
#pragma unroll
        for (int e = 0; e < kColsP; ++e) s[e] = fmaf(s[e], sl2, moff);
        if (masked) {
#pragma unroll
          for (int e = 0; e < kColsP; ++e)
            if (key0 + e > lim) s[e] = -INFINITY;
        }
        float a = 0.f, b = 0.f;
#pragma unroll
        for (int e = 0; e < kColsP; e += 2) {
          s[e] = ex2f(s[e]);
          s[e + 1] = ex2f(s[e + 1]);
          a += s[e];
          b += s[e + 1];
        }
        psum = a + b;
        uint32_t pw[16];
#pragma unroll
        for (int w = 0; w < 8; ++w)
          p_encode4(s[4 * w], s[4 * w + 1], s[4 * w + 2], s[4 * w + 3], pw[w], pw[8 + w]);
        tmem_st16(lane_addr + sb * 128 + col0, pw);           // P_hi then P_lo of these keys
      }
      l = l * alpha + psum;                                   // this group's share
      if (j > 0 && __any_sync(0xffffffffu, rescale)) {
        // O holds the sum up to PV(j - 1): rescale this group's dims once that PV completed.
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars.pv_done[(j - 1) & 1]),
                                               ((j - 1) >> 1) & 1, abort_flag))) {
          alive = false;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {                         // O_hi and O_lo
          const uint32_t col = kOColP + 128 * c + col0;
          uint32_t o[32];
          tmem_ld32(lane_addr + col, o);
          tmem_ld_wait(o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(lane_addr + col, o);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(smem_u32(&bars.p_full[sb]));
    }
    // ---- epilogue: out = v_descale * O / l, lse = (m + log2 l - kShift) ln 2 ---------------------
    // (l is the sum of the groups' shares: they all took the same rescaling decisions)
    if (alive && !exchange(nt, l, false, l)) alive = false;
    if (alive && __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars.pv_done[(nt - 1) & 1]),
                                                   ((nt - 1) >> 1) & 1, abort_flag))) {
      tc_fence_after();
      const float sc = l > 0.f ? vd / l : 0.f;
      const int64_t row = static_cast<int64_t>(q0) + i;
      uint4* dst = reinterpret_cast<uint4*>(prm.out + row * prm.out_stride_tok +
                                            static_cast<int64_t>(h) * prm.out_stride_head +
                                            col0);
      uint32_t o[32], ol[32];
      tmem_ld32(lane_addr + kOColP + col0, o);
      tmem_ld32(lane_addr + kOColP + 128 + col0, ol);
      tmem_ld_wait(o);
      tmem_ld_wait(ol);
      if (valid) {
#pragma unroll
        for (int e = 0; e < 32; ++e)
          o[e] = __float_as_uint(fmaf(__uint_as_float(ol[e]), 0.0625f, __uint_as_float(o[e])));
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const __nv_bfloat162 v2 = __floats2bfloat162_rn(
                __uint_as_float(o[8 * q + 2 * e]) * sc, __uint_as_float(o[8 * q + 2 * e + 1]) * sc);
            w[e] = *reinterpret_cast<const uint32_t*>(&v2);
          }
          dst[q] = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      if (valid && grp == 0 && prm.lse)
        prm.lse[static_cast<int64_t>(h) * prm.total_q + row] =
            l > 0.f ? (m + log2f(l) - kShift) * kLn2 : -INFINITY;
    }
  }

  // ---- teardown ---------------------------------------------------------------------------------
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (*abort_flag && tid == 0) set_status(prm.status, MTPATTN_ERR_TIMEOUT);
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemColsP);
  }
}

// ---- host side ----------------------------------------------------------------------------------

typedef CUresult (*EncodeTiledFnP)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFnP encode_fn_p() {
  static EncodeTiledFnP fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFnP>(f);
  }
  return fn;
}

// [rows][heads][dim] e4m3 bytes as a 3-D tensor (dim, head, row); one box is 128 bytes of the
// head dim (past its end TMA writes zeros) for one head and 128 rows, 128B-swizzled.
bool make_thd_map(CUtensorMap* map, const void* ptr, int64_t rows, int heads, int dim,
                  int64_t stride_tok, int64_t stride_head) {
  EncodeTiledFnP enc = encode_fn_p();
  if (!enc) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(dim), static_cast<cuuint64_t>(heads),
                              static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(stride_head),
                                 static_cast<cuuint64_t>(stride_tok)};
  const cuuint32_t box[3] = {128, 1, 128};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Encoding a tensor map costs microseconds of host time: keep the last few.
struct ThdMapKey {
  const void* ptr;
  int64_t rows, stride_tok, stride_head;
  int heads, dim, device;
  bool operator==(const ThdMapKey& o) const {
    return ptr == o.ptr && rows == o.rows && stride_tok == o.stride_tok &&
           stride_head == o.stride_head && heads == o.heads && dim == o.dim && device == o.device;
  }
};
std::mutex g_thd_mutex;
ThdMapKey g_thd_keys[12];
CUtensorMap g_thd_maps[12];
int g_thd_next = 0;

bool thd_map(CUtensorMap* map, const ThdMapKey& key) {
  std::lock_guard<std::mutex> lock(g_thd_mutex);
  for (int i = 0; i < 12; ++i)
    if (g_thd_keys[i].ptr && g_thd_keys[i] == key) {
      *map = g_thd_maps[i];
      return true;
    }
  if (!make_thd_map(map, key.ptr, key.rows, key.heads, key.dim, key.stride_tok, key.stride_head))
    return false;
  g_thd_keys[g_thd_next] = key;
  g_thd_maps[g_thd_next] = *map;
  g_thd_next = (g_thd_next + 1) % 12;
  return true;
}

bool on_device_p(const void* ptr, int device) {
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

extern "C" int fmha_fwd_fp8_varlen(const void* q, int64_t q_stride_tok, int64_t q_stride_head,
                                   const void* k, int64_t k_stride_tok, int64_t k_stride_head,
                                   const void* v, int64_t v_stride_tok, int64_t v_stride_head,
                                   const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                   int32_t num_seqs, int32_t total_q, int32_t total_k,
                                   int32_t max_seqlen_q, int32_t max_seqlen_k,
                                   int32_t num_q_heads, int32_t num_kv_heads,
                                   const float* q_descale, const float* k_descale,
                                   const float* v_descale, float softmax_scale, int32_t causal,
                                   void* out, int64_t out_stride_tok, int64_t out_stride_head,
                                   float* lse, int32_t* status, void* stream) {
  auto aligned = [](const void* ptr, uintptr_t a) { return reinterpret_cast<uintptr_t>(ptr) % a == 0; };
  if (num_seqs < 0 || total_q < 0 || total_k < 0 || max_seqlen_q < 0 || max_seqlen_k < 0 ||
      num_q_heads <= 0 || num_kv_heads <= 0 || (causal != 0 && causal != 1))
    return MTPATTN_E_ARG;
  if (!q || !k || !v || !cu_seqlens_q || !cu_seqlens_k || !q_descale || !k_descale ||
      !v_descale || !out)
    return MTPATTN_E_ARG;
  if (!isfinite(softmax_scale)) return MTPATTN_E_ARG;
  const int64_t sq[6] = {q_stride_tok, q_stride_head, k_stride_tok, k_stride_head, v_stride_tok,
                         v_stride_head};
  for (int64_t st : sq)
    if (st <= 0 || st % 16 != 0 || st >= (int64_t(1) << 40)) return MTPATTN_E_ARG;
  if (out_stride_tok <= 0 || out_stride_head <= 0 || out_stride_tok % 8 || out_stride_head % 8)
    return MTPATTN_E_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      !aligned(cu_seqlens_q, 4) || !aligned(cu_seqlens_k, 4) || !aligned(q_descale, 4) ||
      !aligned(k_descale, 4) || !aligned(v_descale, 4) || !aligned(lse, 4) || !aligned(status, 4))
    return MTPATTN_E_ARG;
  if (num_q_heads % num_kv_heads) return MTPATTN_E_UNSUPPORTED;
  if (num_seqs == 0 || total_q == 0 || max_seqlen_q == 0) return MTPATTN_OK;
  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess) {
    cudaGetLastError();
    return MTPATTN_E_DEVICE;
  }
  const void* ptrs[] = {q, k, v, cu_seqlens_q, cu_seqlens_k, q_descale, k_descale, v_descale, out};
  for (const void* ptr : ptrs)
    if (!on_device_p(ptr, device)) return MTPATTN_E_DEVICE;
  if ((lse && !on_device_p(lse, device)) || (status && !on_device_p(status, device)))
    return MTPATTN_E_DEVICE;

  PrefillParams prm;
  // An empty key tensor still needs a valid map (no box is ever loaded from it).
  const int64_t krows = total_k > 0 ? total_k : 1;
  if (!thd_map(&prm.tmap_q, {q, total_q, q_stride_tok, q_stride_head, num_q_heads,
                             FMHA_FP8_HEAD_DIM_QK, device}) ||
      !thd_map(&prm.tmap_k, {k, krows, k_stride_tok, k_stride_head, num_kv_heads,
                             FMHA_FP8_HEAD_DIM_QK, device}) ||
      !thd_map(&prm.tmap_v, {v, krows, v_stride_tok, v_stride_head, num_kv_heads,
                             FMHA_FP8_HEAD_DIM_V, device}))
    return MTPATTN_E_ARG;
  prm.cu_q = cu_seqlens_q;
  prm.cu_k = cu_seqlens_k;
  prm.num_seqs = num_seqs;
  prm.total_q = total_q;
  prm.total_k = total_k;
  prm.hq = num_q_heads;
  prm.hkv = num_kv_heads;
  prm.ratio = num_q_heads / num_kv_heads;
  prm.n_qtiles = (max_seqlen_q + kBM - 1) / kBM;
  prm.causal = causal;
  prm.q_descale = q_descale;
  prm.k_descale = k_descale;
  prm.v_descale = v_descale;
  prm.scale_log2 = softmax_scale * kLog2e;
  prm.out = static_cast<__nv_bfloat16*>(out);
  prm.out_stride_tok = out_stride_tok;
  prm.out_stride_head = out_stride_head;
  prm.lse = lse;
  prm.status = status;
  const int64_t grid = static_cast<int64_t>(prm.n_qtiles) * num_q_heads * num_seqs;
  if (grid > 0x7fffffff) return MTPATTN_E_UNSUPPORTED;
  static bool attr_set[64] = {false};
  if (device >= 64) return MTPATTN_E_DEVICE;
  if (!attr_set[device]) {
    if (cudaFuncSetAttribute(fmha_fp8_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemP) != cudaSuccess) {
      cudaGetLastError();
      return MTPATTN_E_LAUNCH;
    }
    attr_set[device] = true;
  }
  fmha_fp8_prefill_kernel<<<static_cast<unsigned>(grid), kThreadsP, kSmemP,
                            static_cast<cudaStream_t>(stream)>>>(prm);
  if (cudaGetLastError() != cudaSuccess) return MTPATTN_E_LAUNCH;
  return MTPATTN_OK;
}
