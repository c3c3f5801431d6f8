// Split-KV main kernel on the sm_100-family tensor cores (tcgen05, TMA, TMEM).
//
// Work items are the (segment s, sequence b, KV head h) triples of the aiter
// PR #5190 page's decomposition ("grid = segments x sequences x kv heads");
// here a persistent grid of one CTA per SM walks them, so the K/V stream of the
// next item starts while the current one finishes.
//
// Roles (192 threads):
//   warp 0   producer: TMA loads of the item's K and V pages, straight from the
//            paged NHD cache through the block table (two 128-byte-wide boxes
//            per page, 128B-swizzled), into 3-stage K and V rings;
//   warp 1   MMA issuer (one thread) and TMEM owner;
//   warps 2-5  softmax group, one TMEM lane each: Q preparation, online
//            softmax, O rescale and the segment epilogue.
//
// Precision.  Both contractions run as e4m3 x e4m3 -> f32 MMAs on the cache
// bytes themselves, so K and V are never converted.  To keep Q and P at bf16
// precision, each is written as the sum of two e4m3 terms:
//   Q:  x = q * 2^a (a per row, so max|x| is in [128, 256)),
//       hi = e4m3(x), lo = e4m3((x - hi) * 16);  x = hi + lo/16 exactly for
//       every element within 2^-13 of the row maximum (a bf16 value has 8
//       significant bits, hi keeps 4 and the remainder fits lo's 4);
//   P:  p * 256 = hi + lo/16 the same way, p in [0, 1].
// The hi and lo rows are stacked into one M = 128 MMA: TMEM lane 32w + t holds
// hi (t < 16) or lo (t >= 16) of query row 16w + (t & 15), so the two halves
// of a row live in lanes t and t ^ 16 of the same warp and are added with one
// shuffle.  S = hi + lo/16 per tile; O = (O_hi + O_lo/16) / 256 at the end.
//
// Tile = 128 keys (8 pages).  TMEM: S double buffer at columns 0 and 128 (the
// tile's P overwrites the first 32 columns of its S buffer, 4 e4m3 per column),
// O at columns 256..511.  QK is 8 MMAs (K = 32 bytes each) with A = stacked Q
// and B = the K tile (both K-major); PV is 4 MMAs with A = P from TMEM and
// B = the V tile read MN-major (dims contiguous).
#include "common.cuh"
#include "sm100.cuh"

#include <cuda_fp8.h>
#include <math.h>

namespace mtpattn {
namespace {

using namespace sm100;

constexpr int kThreads = 192;
constexpr int kTileKeys = 128;
constexpr int kPagesPerTile = kTileKeys / kPage;       // 8
constexpr int kHalfBytes = kTileKeys * 128;            // one 128-byte column half of a tile
constexpr int kTileBytes = 2 * kHalfBytes;             // 32 KB per tensor per tile
constexpr int kStages = 3;
constexpr int kQBytes = 128 * 256;                     // stacked hi/lo Q, two halves of 16 KB
constexpr int kSCols = 128;
constexpr int kOCol = 256;
constexpr int kTmemCols = 512;

// Shared-memory map (offsets from a 1024-byte-aligned base).
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kQBytes;
constexpr int kOffV = kOffK + kStages * kTileBytes;
constexpr int kOffBar = kOffV + kStages * kTileBytes;
constexpr int kSmemBytes = kOffBar + 256 + 1024;       // + barriers + alignment slack

struct TcParams {
  CUtensorMap tmap_k;
  CUtensorMap tmap_v;
  AttnParams a;
  int32_t num_items;
};

struct Bars {
  uint64_t k_full[kStages], k_empty[kStages], v_full[kStages], v_empty[kStages];
  uint64_t s_full[2], p_full[2], pv_done[2];
  uint64_t q_ready, final_mma;
  uint32_t tmem_base;
  int32_t abort;
};
static_assert(sizeof(Bars) <= 256, "barrier block");

// Geometry of one work item, computed identically by every role.
struct Item {
  int s, b, h, L, q0, ql, R, pb, pe, ntiles, err;
};

__device__ __forceinline__ Item item_info(const AttnParams& p, int it, int lane) {
  Item x;
  const int S = p.num_segments;
  x.s = it % S;
  const int rest = it / S;
  x.b = rest % p.num_seqs;
  x.h = rest / p.num_seqs;
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
  if (!x.err) segment_pages(n_pages, S, x.s, &x.pb, &x.pe);
  if (!x.err && x.pe > x.pb) {
    const int32_t* bt = p.block_tables + static_cast<size_t>(x.b) * p.max_pages;
    int bad = 0;
    for (int i = x.pb + lane; i < x.pe; i += 32) {
      const int32_t e = bt[i];
      bad |= (e < 0 || e >= p.num_pages);
    }
    if (__any_sync(0xffffffffu, bad)) x.err |= MTPATTN_ERR_PAGE;
  }
  x.ntiles = x.err ? 0 : (x.pe - x.pb + kPagesPerTile - 1) / kPagesPerTile;
  return x;
}

__device__ __forceinline__ int64_t out_row(const AttnParams& p, const Item& x, int r) {
  const int t = r / p.ratio, g = r - t * p.ratio;
  return static_cast<int64_t>(x.q0 + t) * p.num_q_heads + x.h * p.ratio + g;
}

// Two floats -> two e4m3 codes (RN, saturating), first value in the low byte.
__device__ __forceinline__ uint32_t f2_to_e4m3x2(float a, float b) {
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
}
__device__ __forceinline__ float2 e4m3x2_to_f2(uint32_t v) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(v & 0xFFFF), __NV_E4M3);
  return __half22float2(*reinterpret_cast<__half2*>(&h));
}
// Split x0..x3 into hi codes (4 bytes) and lo codes (4 bytes): x = hi + lo / 16.
__device__ __forceinline__ void split4(float x0, float x1, float x2, float x3, uint32_t& hi,
                                       uint32_t& lo) {
  const uint32_t h01 = f2_to_e4m3x2(x0, x1), h23 = f2_to_e4m3x2(x2, x3);
  const float2 g01 = e4m3x2_to_f2(h01), g23 = e4m3x2_to_f2(h23);
  const uint32_t l01 = f2_to_e4m3x2((x0 - g01.x) * 16.f, (x1 - g01.y) * 16.f);
  const uint32_t l23 = f2_to_e4m3x2((x2 - g23.x) * 16.f, (x3 - g23.y) * 16.f);
  hi = h01 | (h23 << 16);
  lo = l01 | (l23 << 16);
}

__device__ __forceinline__ float pow2f(int e) {  // 2^e for e in [-126, 127]
  return __int_as_float((e + 127) << 23);
}

__global__ void __launch_bounds__(kThreads, 1)
attn_main_tc_kernel(const __grid_constant__ TcParams prm) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Bars& bars = *reinterpret_cast<Bars*>(base + kOffBar);
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
      mbar_init(smem_u32(&bars.p_full[i]), 128);
      mbar_init(smem_u32(&bars.pv_done[i]), 1);
    }
    mbar_init(smem_u32(&bars.q_ready), 128);
    mbar_init(smem_u32(&bars.final_mma), 1);
    bars.abort = 0;
    fence_mbar_init();
  }
  // The V ring must hold finite values before any P = 0 column meets it.
  for (int i = tid; i < (2 * kStages * kTileBytes) / 16; i += kThreads)
    reinterpret_cast<uint4*>(base + kOffK)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;

  if (warp == 0) {
    // ======================================= producer ===========================================
    if (lane == 0) {
      prefetch_tmap(&prm.tmap_k);
      prefetch_tmap(&prm.tmap_v);
    }
    const uint64_t pol = l2_policy_evict_first();
    uint32_t t = 0;  // global tile counter
    for (int it = blockIdx.x; it < prm.num_items && !*abort_flag; it += gridDim.x) {
      const Item x = item_info(p, it, lane);
      if (lane == 0) {
        const int32_t* bt = p.block_tables + static_cast<size_t>(x.b) * p.max_pages;
        for (int j = 0; j < x.ntiles; ++j, ++t) {
          const int pg0 = x.pb + j * kPagesPerTile;
          const int np = min(kPagesPerTile, x.pe - pg0);
          const int st = t % kStages;
          const uint32_t ph = ((t / kStages) & 1) ^ 1;
          if (!mbar_wait(smem_u32(&bars.k_empty[st]), ph, abort_flag)) break;
          const uint32_t kf = smem_u32(&bars.k_full[st]);
          mbar_arrive_expect_tx(kf, np * 2 * 2048);
          const uint32_t kdst = smem_u32(base + kOffK + st * kTileBytes);
          for (int i = 0; i < np; ++i) {
            const int phys = bt[pg0 + i];
            tma_load_4d(kdst + i * 2048, &prm.tmap_k, kf, 0, x.h, 0, phys, pol);
            tma_load_4d(kdst + kHalfBytes + i * 2048, &prm.tmap_k, kf, 128, x.h, 0, phys, pol);
          }
          if (!mbar_wait(smem_u32(&bars.v_empty[st]), ph, abort_flag)) break;
          const uint32_t vf = smem_u32(&bars.v_full[st]);
          mbar_arrive_expect_tx(vf, np * 2 * 2048);
          const uint32_t vdst = smem_u32(base + kOffV + st * kTileBytes);
          for (int i = 0; i < np; ++i) {
            const int phys = bt[pg0 + i];
            tma_load_4d(vdst + i * 2048, &prm.tmap_v, vf, 0, x.h, 0, phys, pol);
            tma_load_4d(vdst + kHalfBytes + i * 2048, &prm.tmap_v, vf, 128, x.h, 0, phys, pol);
          }
        }
      }
      t = __shfl_sync(0xffffffffu, t, 0);
    }
    // Never leave with copies in flight: wait for the last issued tiles of both rings.
    if (lane == 0) {
      for (uint32_t k = 0; k < kStages && k < t; ++k) {
        const uint32_t u = t - 1 - k;
        const uint32_t ph = (u / kStages) & 1;
        volatile int no_abort = 0;
        mbar_wait(smem_u32(&bars.k_full[u % kStages]), ph, &no_abort);
        no_abort = 0;
        mbar_wait(smem_u32(&bars.v_full[u % kStages]), ph, &no_abort);
      }
    }
  } else if (warp == 1) {
    // ======================================= MMA issuer =========================================
    constexpr uint32_t kIdescQK = idesc_e4m3_f32(128, kTileKeys, false);
    constexpr uint32_t kIdescPV = idesc_e4m3_f32(128, kHeadDim, true);
    const uint32_t q_addr = smem_u32(base + kOffQ);
    uint32_t t = 0;
    uint32_t items_run = 0;
    for (int it = blockIdx.x; it < prm.num_items && !*abort_flag; it += gridDim.x) {
      const Item x = item_info(p, it, lane);
      if (x.ntiles == 0) continue;
      if (lane == 0) {
        bool ok = mbar_wait(smem_u32(&bars.q_ready), items_run & 1, abort_flag);
        tc_fence_after();
        auto issue_pv = [&](uint32_t u, bool first) -> bool {
          const int st = u % kStages;
          if (!mbar_wait(smem_u32(&bars.v_full[st]), (u / kStages) & 1, abort_flag)) return false;
          if (!mbar_wait(smem_u32(&bars.p_full[u & 1]), (u >> 1) & 1, abort_flag)) return false;
          tc_fence_after();
          const uint32_t v_addr = smem_u32(base + kOffV + st * kTileBytes);
          const uint32_t p_tmem = tmem + (u & 1) * kSCols;
#pragma unroll
          for (int k = 0; k < kTileKeys / 32; ++k) {
            const uint64_t bd = sdesc_sw128(v_addr + k * 4096, kHalfBytes, 1024);
            mma_f8_ts(tmem + kOCol, p_tmem + 8 * k, bd, kIdescPV, (first && k == 0) ? 0u : 1u);
          }
          mma_commit(smem_u32(&bars.v_empty[st]));
          mma_commit(smem_u32(&bars.pv_done[u & 1]));
          return true;
        };
        for (int j = 0; ok && j < x.ntiles; ++j) {
          const uint32_t u = t + j;
          const int st = u % kStages;
          if (!mbar_wait(smem_u32(&bars.k_full[st]), (u / kStages) & 1, abort_flag)) { ok = false; break; }
          if (u >= 2 && !mbar_wait(smem_u32(&bars.pv_done[u & 1]), ((u - 2) >> 1) & 1, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t k_addr = smem_u32(base + kOffK + st * kTileBytes);
#pragma unroll
          for (int k = 0; k < kHeadDim / 32; ++k) {
            const uint32_t off = (k >> 2) * kHalfBytes + (k & 3) * 32;
            const uint64_t ad = sdesc_sw128(q_addr + (k >> 2) * (kQBytes / 2) + (k & 3) * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(k_addr + off, 16, 1024);
            mma_f8_ss(tmem + (u & 1) * kSCols, ad, bd, kIdescQK, k > 0 ? 1u : 0u);
          }
          mma_commit(smem_u32(&bars.s_full[u & 1]));
          mma_commit(smem_u32(&bars.k_empty[st]));
          if (j > 0 && !issue_pv(u - 1, j == 1)) { ok = false; break; }
        }
        if (ok) issue_pv(t + x.ntiles - 1, x.ntiles == 1);
      }
      t += x.ntiles;
      ++items_run;
    }
    if (lane == 0) {
      mma_commit(smem_u32(&bars.final_mma));
      volatile int no_abort = 0;
      mbar_wait(smem_u32(&bars.final_mma), 0, &no_abort);
    }
  } else {
    // ======================================= softmax group =======================================
    const int quad = warp & 3;                 // TMEM lane quadrant of this warp
    const bool is_hi = lane < 16;
    const int rloc = 16 * quad + (lane & 15);  // query row of this lane
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * quad) << 16);
    const float kd = __ldg(p.k_descale);
    const float vd = __ldg(p.v_descale);
    uint32_t t = 0;
    for (int it = blockIdx.x; it < prm.num_items && !*abort_flag; it += gridDim.x) {
      const Item x = item_info(p, it, lane);
      const bool row_valid = rloc < x.R;
      if (x.err) {
        if (is_hi && row_valid)
          p.lse_part[out_row(p, x, rloc) * p.num_segments + x.s] = __int_as_float(0x7fc00000);
        if (lane == 0 && warp == 2) set_status(p.status, x.err);
        continue;
      }
      if (x.ntiles == 0) {
        if (row_valid) {
          float* o = p.o_part + (out_row(p, x, rloc) * p.num_segments + x.s) * kHeadDim + (is_hi ? 0 : 128);
          for (int d = 0; d < 128; d += 4) *reinterpret_cast<float4*>(o + d) = make_float4(0.f, 0.f, 0.f, 0.f);
          if (is_hi) p.lse_part[out_row(p, x, rloc) * p.num_segments + x.s] = -INFINITY;
        }
        continue;
      }

      // ---- Q: scale the row to [128, 256), split into hi / lo e4m3, write the stacked tile --
      int a_exp = 0;
      {
        const int L32 = 32 * quad + lane;      // A-tile row == TMEM lane
        unsigned char* qrow = base + kOffQ + L32 * 128;
        const __nv_bfloat16* src = nullptr;
        float mx = 0.f;
        if (row_valid) {
          const int tk = rloc / p.ratio, g = rloc - tk * p.ratio;
          src = p.q + static_cast<int64_t>(x.q0 + tk) * p.q_stride_tok +
                static_cast<int64_t>(x.h * p.ratio + g) * p.q_stride_head;
          for (int c = 0; c < kHeadDim; c += 8) {
            const uint4 w = *reinterpret_cast<const uint4*>(src + c);
            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              mx = fmaxf(mx, fabsf(__uint_as_float(ww[k] << 16)));
              mx = fmaxf(mx, fabsf(__uint_as_float(ww[k] & 0xFFFF0000u)));
            }
          }
          if (mx > 0.f) {
            int e;
            frexpf(mx, &e);                      // mx = f * 2^e, f in [0.5, 1)
            a_exp = min(126, max(-126, 8 - e));  // mx * 2^a in [128, 256)
          }
        }
        const float sc = pow2f(a_exp);
#pragma unroll 1
        for (int c = 0; c < 16; ++c) {           // 16 output chunks of 16 codes
          uint32_t out[4] = {0u, 0u, 0u, 0u};
          if (row_valid) {
            const uint4 w0 = *reinterpret_cast<const uint4*>(src + 16 * c);
            const uint4 w1 = *reinterpret_cast<const uint4*>(src + 16 * c + 8);
            const uint32_t ww[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint32_t a0 = ww[2 * k], a1 = ww[2 * k + 1];
              uint32_t hi, lo;
              split4(__uint_as_float(a0 << 16) * sc, __uint_as_float(a0 & 0xFFFF0000u) * sc,
                     __uint_as_float(a1 << 16) * sc, __uint_as_float(a1 & 0xFFFF0000u) * sc, hi, lo);
              out[k] = is_hi ? hi : lo;
            }
          }
          const int half = c >> 3, chunk = c & 7;
          *reinterpret_cast<uint4*>(qrow + half * (kQBytes / 2) + ((chunk ^ (L32 & 7)) * 16)) =
              make_uint4(out[0], out[1], out[2], out[3]);
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(smem_u32(&bars.q_ready));

      const int tk = row_valid ? rloc / p.ratio : 0;
      // last visible key of this row, clipped to the segment's pages
      const int vis_max = row_valid ? min(x.L - x.ql + tk, x.pe * kPage - 1) : -1;
      const float sscale = p.scale_log2 * kd * pow2f(-a_exp);
      float m_run = -INFINITY, l_part = 0.f;

      for (int j = 0; j < x.ntiles; ++j) {
        const uint32_t u = t + j;
        const uint32_t sb = u & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars.s_full[sb]), (u >> 1) & 1, abort_flag))) break;
        tc_fence_after();
        const int key0 = (x.pb + j * kPagesPerTile) * kPage + (is_hi ? 0 : 16);
        float s[64];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t v[32];
          tmem_ld32(lane_addr + sb * kSCols + 32 * c, v);
          tmem_ld_wait(v);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float mine = __uint_as_float(is_hi ? v[i] : v[16 + i]);
            const float send = __uint_as_float(is_hi ? v[16 + i] : v[i]);
            const float other = __shfl_xor_sync(0xffffffffu, send, 16);
            const float comb = is_hi ? fmaf(other, 0.0625f, mine) : fmaf(mine, 0.0625f, other);
            const int key = key0 + 32 * c + i;
            s[16 * c + i] = key <= vis_max ? comb * sscale : -INFINITY;
          }
        }
        float mx = -INFINITY;
#pragma unroll
        for (int i = 0; i < 64; ++i) mx = fmaxf(mx, s[i]);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const float m_new = fmaxf(m_run, mx);
        const bool rescale = m_run != -INFINITY && m_new > m_run;
        const float alpha = rescale ? exp2f(m_run - m_new) : 1.f;
        m_run = m_new;

        // P = 2^(s - m) * 256 as hi / lo e4m3; this lane's 64 keys -> 16 words of each
        uint32_t hiw[16], low[16];
        float psum = 0.f;
#pragma unroll
        for (int w = 0; w < 16; ++w) {
          float pv[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float sv = s[4 * w + k];
            pv[k] = (sv == -INFINITY) ? 0.f : exp2f(sv - m_new);
            psum += pv[k];
          }
          split4(pv[0] * 256.f, pv[1] * 256.f, pv[2] * 256.f, pv[3] * 256.f, hiw[w], low[w]);
        }
        l_part = l_part * alpha + psum;

        // hi lanes gather every hi word of the row, lo lanes every lo word
        uint32_t pw[32];
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t send = is_hi ? low[4 * c + k] : hiw[4 * c + k];
            const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, 16);
            pw[8 * c + k] = is_hi ? hiw[4 * c + k] : recv;
            pw[8 * c + 4 + k] = is_hi ? recv : low[4 * c + k];
          }

        // O may only be touched once the previous tile's PV has completed
        if (j > 0) {
          if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars.pv_done[(u - 1) & 1]), ((u - 1) >> 1) & 1, abort_flag))) break;
          tc_fence_after();
          if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
            for (int c = 0; c < 8; ++c) {
              uint32_t v[32];
              tmem_ld32(lane_addr + kOCol + 32 * c, v);
              tmem_ld_wait(v);
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
              tmem_st32(lane_addr + kOCol + 32 * c, v);
            }
          }
        }
        tmem_st32(lane_addr + sb * kSCols, pw);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(smem_u32(&bars.p_full[sb]));
      }
      if (__any_sync(0xffffffffu, *abort_flag != 0)) break;

      // ---- epilogue: o = v_descale * (O_hi + O_lo / 16) / (256 l), lse = m + log2 l ---------
      const uint32_t ul = t + x.ntiles - 1;
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars.pv_done[ul & 1]), (ul >> 1) & 1, abort_flag))) break;
      tc_fence_after();
      const float l = l_part + __shfl_xor_sync(0xffffffffu, l_part, 16);
      const float oscale = l > 0.f ? vd / (256.f * l) : 0.f;
      float* orow = row_valid ? p.o_part + (out_row(p, x, rloc) * p.num_segments + x.s) * kHeadDim : nullptr;
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        uint32_t v[32];
        tmem_ld32(lane_addr + kOCol + 32 * c, v);
        tmem_ld_wait(v);
        float o[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float mine = __uint_as_float(is_hi ? v[i] : v[16 + i]);
          const float send = __uint_as_float(is_hi ? v[16 + i] : v[i]);
          const float other = __shfl_xor_sync(0xffffffffu, send, 16);
          o[i] = (is_hi ? fmaf(other, 0.0625f, mine) : fmaf(mine, 0.0625f, other)) * oscale;
        }
        if (row_valid) {
          float* dst = orow + 32 * c + (is_hi ? 0 : 16);
#pragma unroll
          for (int i = 0; i < 16; i += 4)
            *reinterpret_cast<float4*>(dst + i) = make_float4(o[i], o[i + 1], o[i + 2], o[i + 3]);
        }
      }
      if (is_hi && row_valid)
        p.lse_part[out_row(p, x, rloc) * p.num_segments + x.s] = l > 0.f ? m_run + log2f(l) : -INFINITY;
      tc_fence_before();
      t += x.ntiles;
    }
  }

  // ---- teardown ------------------------------------------------------------------------------
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

}  // namespace

cudaError_t launch_attn_main(const AttnParams& p, cudaStream_t stream) {
  TcParams prm;
  prm.a = p;
  if (p.num_pages > (int64_t(1) << 31) - 1) return cudaErrorInvalidValue;
  if (!make_cache_map(&prm.tmap_k, p.k_cache, p.num_pages, p.num_kv_heads) ||
      !make_cache_map(&prm.tmap_v, p.v_cache, p.num_pages, p.num_kv_heads))
    return cudaErrorInvalidValue;
  const int64_t items = static_cast<int64_t>(p.num_segments) * p.num_seqs * p.num_kv_heads;
  if (items > (int64_t(1) << 31) - 1) return cudaErrorInvalidValue;
  prm.num_items = static_cast<int32_t>(items);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  static bool attr_set[64] = {false};
  if (!attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(attn_main_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const int sms = device_sm_count(-1);
  if (sms <= 0) return cudaErrorInvalidDevice;
  const int grid = static_cast<int>(items < sms ? items : sms);
  attn_main_tc_kernel<<<grid, kThreads, kSmemBytes, stream>>>(prm);
  return cudaGetLastError();
}

}  // namespace mtpattn
