// fp8 varlen prefill attention, query/key head dim 192 and value head dim 128, on the
// sm_100-family tensor cores (tcgen05, TMA, TMEM): the second workload of the library
// (aiter PR #7375 page, "Summary" and "Changes": e4m3 q/k/v with per-tensor descales, packed
// varlen THD layout, bf16 output, optional log-sum-exp, causal bottom-right or not).
//
// Work: one CTA per (128-query tile, query head, sequence); for a causal call the tiles of a
// head run last-to-first, so the heaviest tiles start first.  Roles (384 threads):
//   warps 0-7   softmax, two sets of four warps: set s takes the key tiles j = s (mod 2) with
//               its own running maximum, sum and O accumulator (split-K inside the CTA), and
//               the two are merged by their log-sum-exps at the end.  Thread t of a set owns
//               query row t (TMEM lane t: warp w reaches lanes 32 (w % 4) .. +31) and all 128
//               keys of the set's tiles, so a row's maximum needs no exchange.  While one set
//               works through a tile the tensor pipe runs the other set's products;
//   warp 8      TMA: the Q tile once, then K tiles (128 keys) and e4m3 V tiles into 2-stage
//               rings (stage s holds set s's tiles);
//   warp 9      MMA: one elected lane issues the tcgen05.mma (kind::f8f6f4 for QK, kind::f16
//               for PV) and the commits, and the warp owns the TMEM allocation;
//   warps 10-11 widen each e4m3 V tile to f16 in shared memory (16 chunks of 16 bytes a
//               thread), the PV operand, off the softmax warps' path.
// 12 warps leave 168 registers a thread: a softmax thread keeps its row's 128 logits.
// A 192-byte q or k row is staged as two 128-byte-swizzled halves of 128 rows; the upper
// half's columns 192..255 lie past the tensor's head dim, and TMA fills them with zeros,
// but QK only runs over bytes 0..191 (6 MMAs of K = 32).  The f16 V tile is 128 keys x 128
// dims, two 128-byte-swizzled atoms of 64 dims, read MN-major as the B operand of PV.
//
// Precision: Q, K and V are the e4m3 inputs themselves (V widened to f16 exactly: every e4m3
// value is an f16 normal or subnormal).  P is rounded once, to f16 (11 significant bits), and
// multiplied with V by the f16 tensor-core product into an f32 accumulator.  A single e4m3 P
// (4 significant bits) would put about 4% of noise on every weight, 0.2-0.3 std of error on
// long rows of comparable logits.
//
// TMEM: S buffer s (set s's tiles) at columns 128 s (fp32), O of set s at 256 + 128 s.  A row's
// P (f16 pairs, keys 2c and 2c + 1 in column c) overwrites columns 0..63 of its S buffer,
// which the thread has read, and PV takes A = P from TMEM.  The MMA warp issues QK(j),
// PV(j-1), QK(j+1), ...: QK(j+2) reuses the buffer whose P(j) PV(j) reads, and the MMAs of
// one thread execute in issue order, so S(j + 2) complete also means PV(j) complete.  PV(j)
// goes out in two halves: keys 0..63 once the set signals that half of P (p_half), while it
// computes keys 64..127, and keys 64..127 at p_full.  The widening warps arrive on the same
// p_half barrier once the tile's f16 V is written, so one wait covers both operands.
//
// The MMA warp issues about 14 products per tile, and the tensor pipe takes each in 80-95
// cycles whatever N (measured: an N = 64 QK costs what an N = 128 one does); every barrier
// poll and tcgen05 fence in its loop leaves the pipe idle meanwhile.  So it fences only where
// another thread's TMEM writes (P) precede the products: a K tile is written and read in the
// async proxy (TMA, tensor cores), ordered by its barrier's transaction count alone.
//
// Online softmax in the log2 domain with a lazy reference m (raised, and O rescaled in TMEM,
// only when a tile's row maximum exceeds it by more than kTau): p_s = 2^(s - m + kShift)
// <= 2^8, and a probability 2^-19 below the row's maximum still keeps all 11 significant bits
// of an f16 (the probability-underflow case of the aiter PR #7375 page's review).
#include "common.cuh"
#include "sm100.cuh"

#include "../../include/fmha_fp8_varlen.h"

#include <cuda_fp8.h>
#include <math.h>

#include <atomic>
#include <mutex>

namespace mtpattn {
namespace {

using namespace sm100;

constexpr int kSets = 2;                        // softmax sets: set s takes the tiles j = s (mod 2)
constexpr int kSetThreads = 128;                // one thread per query row
constexpr int kSoftmaxP = kSets * kSetThreads;
constexpr int kWarpTma = kSoftmaxP / 32, kWarpMma = kWarpTma + 1, kWarpConv = kWarpMma + 1;
constexpr int kConvWarps = 2;
constexpr int kConvThreads = kConvWarps * 32;
constexpr int kThreadsP = kSoftmaxP + 64 + kConvThreads;
constexpr int kBM = 128;                        // query rows per tile
constexpr int kBN = 128;                        // keys per tile
constexpr int kHalfP = 128 * 128;               // one 128-byte-wide half of 128 rows (16 KB)
constexpr int kQTile = 2 * kHalfP;              // 32 KB
constexpr int kKTile = 2 * kHalfP;              // 32 KB per K stage
constexpr int kV8Tile = kHalfP;                 // 16 KB per e4m3 V stage
constexpr int kV16Tile = 2 * kHalfP;            // 32 KB per f16 V stage (two 64-dim atoms)
constexpr int kStagesP = 2;                     // K, e4m3 V and f16 V rings: stage j % 2
constexpr int kOffQP = 0;
constexpr int kOffKP = kOffQP + kQTile;
constexpr int kOffV8P = kOffKP + kStagesP * kKTile;
constexpr int kOffV16P = kOffV8P + kStagesP * kV8Tile;
constexpr int kOffBarP = kOffV16P + kStagesP * kV16Tile;
constexpr int kOffFP = kOffBarP + 256;          // [set][128 rows] final m, then l
constexpr int kLayoutP = kOffFP + 2 * kSets * 128 * 4;
constexpr int kSmemP = kLayoutP + 1024;         // + alignment slack
constexpr int kTmemColsP = 512;
constexpr int kOColP = 256;                     // O of set s at kOColP + 128 s
constexpr float kTau = 3.f;                     // lazy-rescale threshold (log2 units)
constexpr float kShift = 8.f - kTau;            // p_s = 2^(s - m + kShift) <= 2^8
constexpr float kLn2 = 0.6931471805599453f;
static_assert(kStagesP == kSets, "set s owns stage s of every ring and S buffer s");

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
  // p_half: P of keys 0..63 written (the set's 128 threads) and the tile's f16 V written (one
  // arrival per widening warp)
  uint64_t s_full[2], p_half[2], p_full[2], pv_done[2];
  uint64_t final_mma;
  uint64_t fin;                     // both sets' final m and l are published
  uint32_t tmem_base;
  int32_t abort;
};
static_assert(sizeof(PBars) <= 256, "barrier block");

__device__ __forceinline__ float ex2f(float x) {   // 2^x, hardware approximation
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;\n" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float min3f(float a, float b, float c) {
  float d;
  asm("min.f32 %0, %1, %2, %3;\n" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// (a0, a1) * (b0, b1) + (c0, c1), one instruction for the pair
__device__ __forceinline__ void fma_x2(float& a0, float& a1, float b0, float b1, float c0,
                                       float c1) {
  asm("{\n .reg .b64 ra, rb, rc;\n mov.b64 ra, {%0, %1};\n mov.b64 rb, {%2, %3};\n"
      " mov.b64 rc, {%4, %5};\n fma.rn.f32x2 ra, ra, rb, rc;\n mov.b64 {%0, %1}, ra;\n}\n"
      : "+f"(a0), "+f"(a1)
      : "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}
__device__ __forceinline__ void add_x2(float& a0, float& a1, float b0, float b1) {
  asm("{\n .reg .b64 ra, rb;\n mov.b64 ra, {%0, %1};\n mov.b64 rb, {%2, %3};\n"
      " add.rn.f32x2 ra, ra, rb;\n mov.b64 {%0, %1}, ra;\n}\n"
      : "+f"(a0), "+f"(a1)
      : "f"(b0), "f"(b1));
}
// two f32 -> f16x2 (p0 in the low half: the lower K index of a TMEM A-operand cell)
__device__ __forceinline__ uint32_t f16x2_of(float p0, float p1) {
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;\n" : "=r"(d) : "f"(p1), "f"(p0));
  return d;
}
// four e4m3 codes (lowest byte first) -> two f16x2 words, exactly
__device__ __forceinline__ void widen4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n .reg .b16 a, b;\n mov.b32 {a, b}, %2;\n cvt.rn.f16x2.e4m3x2 %0, a;\n"
      " cvt.rn.f16x2.e4m3x2 %1, b;\n}\n"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// 32 lanes x 16 columns of 32 bits: thread t of the warp gets lane (base lane + t).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%16];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld16_wait(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;\n"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}

// tcgen05.mma kind::f16 (f16 x f16 -> f32), A from tensor memory, B from shared memory.
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Instruction descriptor of kind::f16 with f16 A and B and an f32 accumulator: the fields of
// the kind::f8f6f4 descriptor, where format code 0 is f16 (and e4m3 there).
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N, bool b_mn_major) {
  return idesc_e4m3_f32(M, N, b_mn_major);
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
      mbar_init(smem_u32(&bars.v_empty[i]), kConvWarps);        // one arrival per converter warp
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bars.s_full[i]), 1);
      mbar_init(smem_u32(&bars.p_half[i]), kSetThreads + kConvWarps);
      mbar_init(smem_u32(&bars.p_full[i]), kSetThreads);
      mbar_init(smem_u32(&bars.pv_done[i]), 1);
    }
    mbar_init(smem_u32(&bars.final_mma), 1);
    mbar_init(smem_u32(&bars.fin), kSoftmaxP);
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
#ifdef MTPATTN_TEST_STALL
        // Test builds only: CTA 0 never issues its first V tile, so the widening warps' wait
        // for it runs out and the call winds down with MTPATTN_ERR_TIMEOUT.
        if (blockIdx.x == 0 && j == 0) continue;
#endif
        mbar_arrive_expect_tx(vb, kV8Tile);
        tma_load_3d(smem_u32(base + kOffV8P + st * kV8Tile), &prm.tmap_v, vb, 0, hk, k0 + j * kBN);
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
    constexpr uint32_t kIdescPV = idesc_f16_f32(kBM, 128, true);
    const uint64_t q_desc = sdesc_sw128(smem_u32(base + kOffQP), 16, 1024);
    const uint64_t k_desc = sdesc_sw128(smem_u32(base + kOffKP), 16, 1024);
    // f16 V: 64-dim atoms kHalfP apart (MN direction), 8-key groups 1024 bytes apart
    const uint64_t v_desc = sdesc_sw128(smem_u32(base + kOffV16P), kHalfP, 1024);
    const bool leader = elect_one();
    auto wait_all = [&](uint64_t& bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(smem_u32(&bar), parity, abort_flag));
    };
    auto issue_pv = [&](int u) -> bool {
      // P(u) in TMEM and the f16 V(u) in shared memory (both behind p_half); the products of
      // keys 0..63 go out as soon as their half of P is written, while the softmax works on
      // keys 64..127
      const uint32_t p_tmem = tmem + (u & 1) * 128;
      const uint32_t v_off = (u & 1) * kV16Tile;
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        if (!wait_all(half == 0 ? bars.p_half[u & 1] : bars.p_full[u & 1], (u >> 1) & 1))
          return false;
        tc_fence_after();
        if (leader) {
          // keys 16 k .. 16 k + 15: P at columns 8 k .. 8 k + 7, V rows 16 k .. 16 k + 15
          // (128 bytes each in both atoms); the set's own accumulator, first written by its
          // first tile (u < 2)
#pragma unroll
          for (int k = 4 * half; k < 4 * half + 4; ++k)
            mma_f16_ts(tmem + kOColP + 128 * (u & 1), p_tmem + 8 * k,
                       v_desc + ((v_off + k * 2048) >> 4), kIdescPV, (u > 1 || k > 0) ? 1u : 0u);
          if (half == 1) mma_commit(smem_u32(&bars.pv_done[u & 1]));
        }
        __syncwarp();
      }
      return true;
    };
    bool ok = wait_all(bars.q_full, 0);
    for (int j = 0; ok && j < nt; ++j) {
      const int st = j % kStagesP;
      if (!wait_all(bars.k_full[st], (j / kStagesP) & 1)) { ok = false; break; }
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
  } else if (warp >= kWarpConv) {
    // ===================================== V widening ============================================
    // Thread c handles chunk slot vc = c % 8 of keys c / 8 + 8 i (i = 0..15), all with the same
    // key % 8, hence the same logical chunk vcl (dims 16 vcl .. + 15, swizzled) and the same
    // positions of its two f16 halves in the 64-dim atoms.
    const int ct = tid - kWarpConv * 32;
    const int vk = ct >> 3, vc = ct & 7;
    const int vcl = vc ^ (vk & 7);
    const uint32_t v8_off = vk * 128 + vc * 16;
    const uint32_t v16_off0 = (vcl >> 2) * kHalfP + vk * 128 + (((2 * (vcl & 3)) ^ (vk & 7)) << 4);
    const uint32_t v16_off1 = (vcl >> 2) * kHalfP + vk * 128 + (((2 * (vcl & 3) + 1) ^ (vk & 7)) << 4);
    for (int j = 0; j < nt; ++j) {
      const int st = j & 1;
      // V(j) landed, and the f16 slot is free once PV(j - 2) completed
      if (!__all_sync(0xffffffffu,
                      mbar_wait(smem_u32(&bars.v_full[st]), (j >> 1) & 1, abort_flag) &&
                          (j < 2 || mbar_wait(smem_u32(&bars.pv_done[st]), ((j - 2) >> 1) & 1,
                                              abort_flag))))
        break;
      tc_fence_after();
      const unsigned char* src = base + kOffV8P + st * kV8Tile + v8_off;
      unsigned char* dst = base + kOffV16P + st * kV16Tile;
      // all loads first: a store may alias a later load as far as the compiler knows, which
      // would serialise load, widen and store chunk by chunk
      uint4 a[16];
#pragma unroll
      for (int c = 0; c < 16; ++c) a[c] = *reinterpret_cast<const uint4*>(src + c * 8 * 128);
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        uint4 w0, w1;
        widen4(a[c].x, w0.x, w0.y);
        widen4(a[c].y, w0.z, w0.w);
        widen4(a[c].z, w1.x, w1.y);
        widen4(a[c].w, w1.z, w1.w);
        *reinterpret_cast<uint4*>(dst + v16_off0 + c * 8 * 128) = w0;
        *reinterpret_cast<uint4*>(dst + v16_off1 + c * 8 * 128) = w1;
      }
      fence_proxy_async_smem();        // visible to the tensor cores once p_half is observed
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&bars.p_half[st]));      // tile j belongs to set j % 2 = st
        mbar_arrive(smem_u32(&bars.v_empty[st]));
      }
    }
  } else {
    // ===================================== softmax (rows) ========================================
    const int set = warp >> 2;                                // tiles j = set (mod 2), S buffer set
    const int quad = warp & 3;                                // TMEM lane quarter
    const int r = 32 * quad + lane;                           // query row of the tile, TMEM lane
    const int i = i0 + r;
    const bool valid = i < Lq;
    // last key index row i may see (within the sequence)
    const int lim = !valid ? -1 : (prm.causal ? min(Lk - 1, i + Lk - Lq) : Lk - 1);
    const float sl2 = prm.scale_log2 * __ldg(prm.q_descale) * __ldg(prm.k_descale);
    const float vd = __ldg(prm.v_descale);
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * quad) << 16);
    const uint32_t s_addr = lane_addr + set * 128;            // the set's S (then P) columns
    const uint32_t o_addr = lane_addr + kOColP + set * 128;
    float* fin_m = reinterpret_cast<float*>(base + kOffFP);   // [set][row]
    float* fin_l = fin_m + kSets * 128;
    float m = -INFINITY, l = 0.f;
    bool alive = true;
    int u = 0;                                                // the set's own tile count
    for (int j = set; j < nt; j += kSets, ++u) {
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars.s_full[set]), u & 1, abort_flag))) {
        alive = false;
        break;
      }
      tc_fence_after();
      const int key0 = j * kBN;
      const bool masked = key0 + kBN - 1 > lim;               // some key past the row's reach
      // the row's 128 raw logits <q, k> (unscaled), one TMEM round trip
      float s[kBN];
      {
        uint32_t v0[32], v1[32], v2[32], v3[32];
        tmem_ld32(s_addr, v0);
        tmem_ld32(s_addr + 32, v1);
        tmem_ld32(s_addr + 64, v2);
        tmem_ld32(s_addr + 96, v3);
        tmem_ld_wait(v0);
        tmem_ld_wait(v1);
        tmem_ld_wait(v2);
        tmem_ld_wait(v3);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          s[e] = __uint_as_float(v0[e]);
          s[32 + e] = __uint_as_float(v1[e]);
          s[64 + e] = __uint_as_float(v2[e]);
          s[96 + e] = __uint_as_float(v3[e]);
        }
      }
      if (masked) {                                           // out of the maximum below
#pragma unroll
        for (int e = 0; e < kBN; ++e)
          if (key0 + e > lim) s[e] = sl2 >= 0.f ? -INFINITY : INFINITY;
      }
      // the largest scaled logit: sl2 times the largest (sl2 >= 0) or smallest raw one
      float hm;
      if (sl2 >= 0.f) {
        float a = fmaxf(s[0], s[1]), c = fmaxf(s[2], s[3]);
#pragma unroll
        for (int e = 4; e < kBN; e += 4) {
          a = max3f(a, s[e], s[e + 1]);
          c = max3f(c, s[e + 2], s[e + 3]);
        }
        hm = fmaxf(a, c);
      } else {
        float a = fminf(s[0], s[1]), c = fminf(s[2], s[3]);
#pragma unroll
        for (int e = 4; e < kBN; e += 4) {
          a = min3f(a, s[e], s[e + 1]);
          c = min3f(c, s[e + 2], s[e + 3]);
        }
        hm = fminf(a, c);
      }
      float mx = hm * sl2;                                    // the tile's row maximum
      if (mx != mx) mx = -INFINITY;                           // 0 * inf (sl2 = 0, masked)
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
      if (u > 0 && __any_sync(0xffffffffu, rescale)) {
        // the set's O holds its sum up to PV(j - 2), complete: QK(j) was issued after it; the
        // first products of this tile may start once P's first half is signalled below
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {                      // 16 columns at a time: the row's
          uint32_t o[16];                                 // logits are live meanwhile
          tmem_ld16(o_addr + 16 * c, o);
          tmem_ld16_wait(o);
#pragma unroll
          for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st16(o_addr + 16 * c, o);
        }
      }
      // p = 2^(sl2 s + kShift - m), masked keys 2^-inf = 0; P (f16 pairs) over the S columns,
      // 32 keys (16 columns) at a time; keys 0..63 are signalled on their own (p_half)
      float a0 = 0.f, a1 = 0.f, c0 = 0.f, c1 = 0.f;
#pragma unroll
      for (int h4 = 0; h4 < 4; ++h4) {
#pragma unroll
        for (int e = 32 * h4; e < 32 * h4 + 32; e += 2) fma_x2(s[e], s[e + 1], sl2, sl2, moff, moff);
        if (masked) {
#pragma unroll
          for (int e = 32 * h4; e < 32 * h4 + 32; ++e)
            if (key0 + e > lim) s[e] = -INFINITY;
        }
        uint32_t pw[16];
#pragma unroll
        for (int e = 32 * h4; e < 32 * h4 + 32; e += 4) {
          s[e] = ex2f(s[e]);
          s[e + 1] = ex2f(s[e + 1]);
          s[e + 2] = ex2f(s[e + 2]);
          s[e + 3] = ex2f(s[e + 3]);
          add_x2(a0, a1, s[e], s[e + 1]);
          add_x2(c0, c1, s[e + 2], s[e + 3]);
          pw[(e - 32 * h4) / 2] = f16x2_of(s[e], s[e + 1]);
          pw[(e - 32 * h4) / 2 + 1] = f16x2_of(s[e + 2], s[e + 3]);
        }
        tmem_st16(s_addr + 16 * h4, pw);
        if (h4 == 1) {
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(smem_u32(&bars.p_half[set]));
        }
      }
      l = l * alpha + ((a0 + c0) + (a1 + c1));
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(smem_u32(&bars.p_full[set]));
    }
    // ---- epilogue: merge the two sets' (m, l, O); out = v_descale * O / l,
    //      lse = (m + log2 l - kShift) ln 2 ----------------------------------------------------------
    if (alive) {
      fin_m[set * 128 + r] = m;
      fin_l[set * 128 + r] = l;
    }
    mbar_arrive(smem_u32(&bars.fin));
    const int n0 = (nt + 1) / 2, n1 = nt / 2;                 // tiles of set 0 and set 1
    alive = alive && __all_sync(0xffffffffu,
                                mbar_wait(smem_u32(&bars.fin), 0, abort_flag) &&
                                    mbar_wait(smem_u32(&bars.pv_done[0]), (n0 - 1) & 1, abort_flag) &&
                                    (n1 == 0 || mbar_wait(smem_u32(&bars.pv_done[1]), (n1 - 1) & 1,
                                                          abort_flag)));
    if (alive) {
      tc_fence_after();
      const float m0 = fin_m[r], l0 = fin_l[r];
      const float m1 = n1 > 0 ? fin_m[128 + r] : -INFINITY, l1 = n1 > 0 ? fin_l[128 + r] : 0.f;
      const bool use0 = l0 > 0.f, use1 = l1 > 0.f;            // l > 0 implies a finite m
      const float M = use0 && use1 ? fmaxf(m0, m1) : (use0 ? m0 : m1);
      const float w0 = use0 ? ex2f(m0 - M) : 0.f, w1 = use1 ? ex2f(m1 - M) : 0.f;
      const float L = w0 * l0 + w1 * l1;
      const float sc = L > 0.f ? vd / L : 0.f;
      // this thread writes dims 64 set .. 64 set + 63 of its row, 16 at a time
      const uint32_t dcol = 64 * set;
      const int64_t row = static_cast<int64_t>(q0) + i;
      uint4* dst = reinterpret_cast<uint4*>(prm.out + row * prm.out_stride_tok +
                                            static_cast<int64_t>(h) * prm.out_stride_head + dcol);
      const float s0 = w0 * sc, s1 = w1 * sc;
#pragma unroll 1
      for (int hh = 0; hh < 4; ++hh) {
        uint32_t oa[16], ob[16];
        tmem_ld16(lane_addr + kOColP + dcol + 16 * hh, oa);
        tmem_ld16(lane_addr + kOColP + 128 + dcol + 16 * hh, ob);
        tmem_ld16_wait(oa);
        tmem_ld16_wait(ob);
        if (valid) {
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int d = 8 * q + 2 * e;
              // a set with no weight contributes nothing (its accumulator may be unwritten)
              const float x0 = (use0 ? __uint_as_float(oa[d]) * s0 : 0.f) +
                               (use1 ? __uint_as_float(ob[d]) * s1 : 0.f);
              const float x1 = (use0 ? __uint_as_float(oa[d + 1]) * s0 : 0.f) +
                               (use1 ? __uint_as_float(ob[d + 1]) * s1 : 0.f);
              const __nv_bfloat162 v2 = __floats2bfloat162_rn(x0, x1);
              w[e] = *reinterpret_cast<const uint32_t*>(&v2);
            }
            dst[2 * hh + q] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
      if (valid && set == 0 && prm.lse)
        prm.lse[static_cast<int64_t>(h) * prm.total_q + row] =
            L > 0.f ? (M + log2f(L) - kShift) * kLn2 : -INFINITY;
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
  if (num_seqs == 0 || total_q == 0) return MTPATTN_OK;
  if (max_seqlen_q == 0) return MTPATTN_E_ARG;       // queries, but none per sequence
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
  static std::atomic<bool> attr_set[64];   // per device; setting it twice is harmless
  if (device >= 64) return MTPATTN_E_DEVICE;
  if (!attr_set[device].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(fmha_fp8_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemP) != cudaSuccess) {
      cudaGetLastError();
      return MTPATTN_E_LAUNCH;
    }
    attr_set[device].store(true, std::memory_order_release);
  }
  fmha_fp8_prefill_kernel<<<static_cast<unsigned>(grid), kThreadsP, kSmemP,
                            static_cast<cudaStream_t>(stream)>>>(prm);
  if (cudaGetLastError() != cudaSuccess) return MTPATTN_E_LAUNCH;
  return MTPATTN_OK;
}
