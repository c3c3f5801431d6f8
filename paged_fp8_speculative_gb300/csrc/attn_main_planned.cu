// Split-KV main kernel with planned scheduling (tcgen05, TMA, TMEM on the sm_100 family).
//
// The roles, the hi/lo e4m3 precision scheme, the TMEM layout, the online softmax and the
// per-role loops are shared with the chunked kernel (attn_main_common.cuh, attn_main_body.inc);
// this file differs in how pieces are laid out and in how a CTA finds its piece.  Each kernel
// is compiled in its own translation unit: with both ways of scheduling in one source (a
// template over the scheduling) the hot loops ran measurably slower, a few percent at
// 16 x 35k tokens.
//
// Scheduling.  The chunked kernel cuts every (sequence, KV head) unit as if it held
// max_pages pages, which leaves SMs idle on ragged batches.  When the caller leaves S to the
// library, the plan may also give a long unit more than S pieces if short units use fewer of
// the workspace's rows x S partial slots (the slot pool, see AttnParams and plan_piece).  Here the kernel first reads
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
#include "attn_main_common.cuh"

#include <algorithm>
#include <atomic>

namespace mtpattn {
namespace {

using namespace sm100;
using namespace mainkern;

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


// Position in this CTA's walk: chunk k and unit u (unit = h * num_seqs + b).
struct Cursor {
  int64_t k, u;
  int s, pu, C;            // planned scheduling: slot, pieces of the unit, pages per piece
  int b, h;                // planned scheduling: the unit's sequence and KV head
  int L, q0, q1;           // planned scheduling: the unit's seq_lens and cu_seqlens_q entries
  int pool, off;           // slot-pool layout, and the unit's first row-slot there
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

// ceil(x / c) for 0 <= x < 2^22 and 2 <= c < 2^22 with integer operations only, given
// m = ceil(2^32 / c) (magic_of): the estimate umulhi(x + c - 1, m) is at most one too large.
__device__ __forceinline__ uint32_t magic_of(int c) { return 0xFFFFFFFFu / static_cast<uint32_t>(c) + 1u; }
__device__ __forceinline__ int ceil_div_magic(int x, int c, uint32_t m) {
  const uint32_t y = static_cast<uint32_t>(x + c - 1);
  uint32_t q = __umulhi(y, m);
  if (q * static_cast<uint32_t>(c) > y) --q;
  return static_cast<int>(q);
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
    c.pool = c.off = 0;
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
  // Unequal lengths.  This path runs once per call on every SM, so it is written for small
  // code rather than for few instructions: its loops stay rolled over the lane's unit slots
  // (fetching cold straight-line code cost more than the arithmetic), on copies of the
  // per-slot values that may live in local memory.
  int nl[8], Rl[8], pl[8], Ll[8], q0l[8], q1l[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    nl[i] = n[i];
    Ll[i] = Lv[i];
    q0l[i] = q0v[i];
    q1l[i] = q1v[i];
  }
  auto warp_sum = [](int x) -> int {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
  };
  int total = 0;
#pragma unroll 1
  for (int i = 0; i < nb; ++i) total += nl[i];
  total = warp_sum(total);
  // sum_v ceil(n_v / c), and (weighted by the units' query rows) the row-slots it takes
  auto count = [&](int c, int& rows_slots) -> int {
    const float inv = 1.f / static_cast<float>(c);
    int t = 0, w = 0;
#pragma unroll 1
    for (int i = 0; i < nb; ++i)
      if (nl[i] > 0) {
        const int q = ceil_div_inv(nl[i], c, inv);
        t += q;
        w += Rl[i] * q;
      }
    rows_slots = warp_sum(w);
    return warp_sum(t);
  };
#pragma unroll 1
  for (int i = 0; i < nb; ++i) {
    const int ql = q1l[i] - q0l[i];
    Rl[i] = (nl[i] > 0 && q0l[i] >= 0 && q1l[i] <= p.total_q && ql >= 1 && ql <= kMaxQLen)
                ? ql * p.ratio : 0;
  }
  if (U <= 32) {
    // At most one unit per lane: each lane tests its own candidate piece size against every
    // unit (the units' values come by shuffle inside a rolled loop) and a ballot gives the
    // first candidate that passes, so a search over N values takes log32(N) rounds and no
    // chains of warp reductions.  Same plan as the loop below.
    const bool pool_ok = p.slot_pool && G <= 256;
    const int n_own = nl[0], R_own = Rl[0];
    const int hi0s = max(maxn, 1);
    const int lo_gs = max((total + G - 1) / G, min(kPagesPerTile, hi0s));
    const int hi_gs = G > U ? min(hi0s, (total + (G - U) - 1) / (G - U)) : hi0s;
    const int lo_ss = min(max(lo_gs, (maxn + S - 1) / S), hi0s);
    // The smallest C in [lo_gs (lo_ss without the pool), max(lo_ss, hi_gs)] with
    // sum_v ceil(n_v / C) <= G and either max_v ceil(n_v / C) <= S (the row-major slots) or,
    // with the slot pool allowed, sum_v R_v ceil(n_v / C) within the pool.  All three sums
    // fall as C grows, so the condition holds from some C on (the top of the range passes)
    // and one search finds it; the pool is used only where the S cap is what fails (max
    // pieces > S, below).  This is the C of the two searches below (S cap, then pool).
    int clo = pool_ok ? lo_gs : lo_ss;
    int chi = max(lo_ss, hi_gs);
    while (clo < chi) {
      const int step = (chi - clo + 32) / 32;                     // ceil((chi - clo + 1) / 32)
      const int c = min(clo + (lane + 1) * step - 1, chi);        // lane 31's candidate is chi
      const bool trivial = c >= chi || c >= maxn;                  // passes by construction
      const uint32_t mg = magic_of(max(c, 2));
      int t = 0, w = 0, mx = 0;
#pragma unroll 1
      for (int v = 0; v < U; ++v) {                               // every lane, uniformly
        const int nv = __shfl_sync(0xffffffffu, n_own, v);
        const int rv = __shfl_sync(0xffffffffu, R_own, v);
        const int q = nv > 0 ? ceil_div_magic(nv, max(c, 2), mg) : 0;
        t += q;
        w += rv * q;
        mx = max(mx, q);
      }
      const bool ok = trivial || (t <= G && (mx <= S || (pool_ok && w <= p.pool_cap)));
      const int f = __ffs(__ballot_sync(0xffffffffu, ok)) - 1;
      const int cf = min(clo + (f + 1) * step - 1, chi);
      clo = f == 0 ? clo : min(clo + f * step - 1, chi) + 1;
      chi = cf;
    }
    const int Cs = clo;
    const int p_own = (lane < U && n_own > 0) ? (Cs >= n_own ? 1 : ceil_div_magic(n_own, Cs, magic_of(Cs))) : 0;
    const int npieces = warp_sum(p_own);
    int maxp = p_own;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) maxp = max(maxp, __shfl_xor_sync(0xffffffffu, maxp, o));
    const bool pools = pool_ok && maxp > S;
    Cursor c;
    c.C = Cs;
    c.s = 0;
    c.pu = 0;
    c.u = 0;
    c.b = c.h = 0;
    c.pool = pools ? 1 : 0;
    c.off = 0;
    c.L = c.q0 = c.q1 = 0;
    const int k = blockIdx.x;
    if (k >= npieces) {                      // more CTAs than pieces: nothing for this one
      c.k = prm.num_chunks;
      return c;
    }
    // slot-major: the slot is the largest sl with sum_v min(p_v, sl) <= k
    auto before = [&](int sl) -> int {
      int t = 0;
#pragma unroll 1
      for (int v = 0; v < U; ++v) t += min(__shfl_sync(0xffffffffu, p_own, v), sl);
      return t;
    };
    int lo = 0, hi = maxp - 1;               // before(0) = 0 <= k
    while (lo < hi) {                        // largest sl in [lo, hi] with before(sl) <= k
      const int step = (hi - lo + 32) / 32;
      const int cand = min(lo + lane * step, hi);
      const int f = 31 - __clz(__ballot_sync(0xffffffffu, before(cand) <= k));   // lane 0 passes
      const int cf = min(lo + f * step, hi);
      hi = f == 31 ? hi : min(lo + (f + 1) * step, hi) - 1;
      lo = cf;
    }
    const int slot = lo;
    int r = k;                               // minus the pieces of slots below: sum_v min(p_v, slot)
#pragma unroll 1
    for (int v = 0; v < U; ++v) r -= min(__shfl_sync(0xffffffffu, p_own, v), slot);
    uint32_t m = __ballot_sync(0xffffffffu, p_own > slot);
    for (int q = 0; q < r; ++q) m &= m - 1;  // drop the r lowest set bits
    const int u = __ffs(m) - 1;
    c.k = k;
    c.u = u;
    c.s = slot;
    c.pu = __shfl_sync(0xffffffffu, p_own, u);
    c.L = __shfl_sync(0xffffffffu, Ll[0], u);
    c.q0 = __shfl_sync(0xffffffffu, q0l[0], u);
    c.q1 = __shfl_sync(0xffffffffu, q1l[0], u);
    c.h = div_inv(u, B, prm.inv_seqs);
    c.b = u - c.h * B;
    if (pools) c.off = warp_sum(lane < u ? R_own * p_own : 0);
    return c;
  }
  // The smallest C with sum_v ceil(n_v / C) <= G (it lies in [ceil(total / G),
  // ceil(total / (G - U))], since that sum is at most total / C + U), no piece below one
  // 128-key tile, and at most S pieces per unit (C >= ceil(maxn / S)) -- or, with the slot
  // pool allowed (the caller let the library choose S), with the rows x pieces within the
  // pool instead of the S cap, when that gives a smaller C (the S cap was binding).
  const int hi0 = max(maxn, 1);
  const int lo_g = max((total + G - 1) / G, min(kPagesPerTile, hi0));
  const int hi_g = G > U ? min(hi0, (total + (G - U) - 1) / (G - U)) : hi0;
  const int lo_s = min(max(lo_g, (maxn + S - 1) / S), hi0);
  const bool pool_ok = p.slot_pool && G <= 256;
  int C = 0;
  bool pool = false;
#pragma unroll 1
  for (int pass = 0; pass < 2; ++pass) {
    // pass 0: the S cap; pass 1 (slot pool): the row-slot capacity, below pass 0's C
    int lo = pass == 0 ? lo_s : lo_g;
    int hi = pass == 0 ? max(lo_s, hi_g) : C - 1;
    if (pass == 1 && (!pool_ok || hi < lo)) break;
    if (pass == 1) {                          // is anything below pass 0's C feasible at all?
      int w;
      if (count(hi, w) > G || w > p.pool_cap) break;
    }
    while (lo < hi) {
      const int mid = (lo + hi) / 2;
      int w;
      const bool ok = count(mid, w) <= G && (pass == 0 || w <= p.pool_cap);
      if (ok) hi = mid;
      else lo = mid + 1;
    }
    C = lo;
    pool = pass == 1;
  }
  int maxp = 0, npieces = 0;
  {
    const float invC = 1.f / static_cast<float>(C);
#pragma unroll 1
    for (int i = 0; i < 8; ++i) {
      pl[i] = (i < nb && nl[i] > 0) ? ceil_div_inv(nl[i], C, invC) : 0;
      maxp = max(maxp, pl[i]);
      npieces += pl[i];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) maxp = max(maxp, __shfl_xor_sync(0xffffffffu, maxp, o));
    npieces = warp_sum(npieces);
  }
  auto before = [&](int sl) -> int {         // pieces of slots below sl: sum_v min(p_v, sl)
    int t = 0;
#pragma unroll 1
    for (int i = 0; i < nb; ++i) t += min(pl[i], sl);
    return warp_sum(t);
  };
  Cursor c;
  c.C = C;
  c.s = 0;
  c.pu = 0;
  c.u = 0;
  c.b = c.h = 0;
  c.pool = pool ? 1 : 0;
  c.off = 0;
  c.L = c.q0 = c.q1 = 0;
  const int k = blockIdx.x;
  if (k >= npieces) {                        // more CTAs than pieces: nothing for this one
    c.k = prm.num_chunks;
    return c;
  }
  int slo = 0, shi = maxp - 1;               // largest slot sl with before(sl) <= k
  int bslo = 0;                              // before(slo)
  while (slo < shi) {
    const int mid = (slo + shi + 1) / 2;
    const int bm = before(mid);
    if (bm <= k) {
      slo = mid;
      bslo = bm;
    } else {
      shi = mid - 1;
    }
  }
  int r = k - bslo;                          // the r-th unit (in order) that has slot slo
  int u = -1, pu_u = 0;
#pragma unroll 1
  for (int i = 0; i < nb && u < 0; ++i) {
    const uint32_t m = __ballot_sync(0xffffffffu, pl[i] > slo);
    const int cnt = __popc(m);
    if (r < cnt) {
      uint32_t mm = m;
      for (int q = 0; q < r; ++q) mm &= mm - 1;        // drop the r lowest set bits
      const int ln = __ffs(mm) - 1;
      u = ln + 32 * i;
      pu_u = __shfl_sync(0xffffffffu, pl[i], ln);
      c.L = __shfl_sync(0xffffffffu, Ll[i], ln);
      c.q0 = __shfl_sync(0xffffffffu, q0l[i], ln);
      c.q1 = __shfl_sync(0xffffffffu, q1l[i], ln);
    } else {
      r -= cnt;
    }
  }
  c.k = k;
  c.u = u;
  c.s = slo;
  c.pu = pu_u;
  c.h = div_inv(u, B, prm.inv_seqs);
  c.b = u - c.h * B;
  if (pool) {                                // the unit's first row-slot: sum_{v < u} R_v p_v
    int t = 0;
#pragma unroll 1
    for (int i = 0; i < nb; ++i)
      if (lane + 32 * i < u) t += Rl[i] * pl[i];
    c.off = warp_sum(t);
  }
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
  int pool;    // slot-pool layout (see AttnParams)
  int off;     // slot pool: the unit's first row-slot
  bool last;   // the unit's last piece: it also marks the unit's unused slots empty
};

__device__ __forceinline__ Item item_info(const TcParams& prm, const Cursor& c, int lane) {
  const AttnParams& p = prm.a;
  Item x;
  x.pieces = c.pu;                         // everything comes with the plan
  x.pool = c.pool;
  x.off = c.off;
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


// Split slots.  Row-major (the default): the S slots of output row rho at rho * S + s.  Slot
// pool: piece s of unit v writes row r of the unit at row-slot off_v + r * p_v + s of the
// pool (see AttnParams), and its first piece writes the row's redirect for the reduce.
__device__ __forceinline__ float* lse_slot(const AttnParams& p, const Item& x, int r) {
  if (x.pool) return p.pool_lse + x.off + r * x.pieces + x.s;
  return p.lse_part + out_row(p, x, r) * p.num_segments + x.s;
}
__device__ __forceinline__ float* o_slot(const AttnParams& p, const Item& x, int r) {
  if (x.pool) return p.o_part + static_cast<int64_t>(x.off + r * x.pieces + x.s) * kHeadDim;
  return p.o_part + (out_row(p, x, r) * p.num_segments + x.s) * kHeadDim;
}
__device__ __forceinline__ void close_unit_rows(const AttnParams& p, const Item& y, int r) {
  float* row = p.lse_part + out_row(p, y, r) * p.num_segments;
  if (y.pool) {
    if (y.s == 0) {
      row[0] = __uint_as_float(kPoolMarker);
      row[1] = __int_as_float(y.off + r * y.pieces);
      row[2] = __int_as_float(y.pieces);
    }
  } else if (y.last) {
    for (int s2 = y.s + 1; s2 < p.num_segments; ++s2) row[s2] = -INFINITY;
  }
}

// The CTA's piece.  The K producer warp plans and publishes the plan in the barrier block; the
// other warps wait for it there and read it.
__device__ __forceinline__ Cursor first_cursor_of(const TcParams& prm, Bars& bars, int warp,
                                                  int lane, volatile int* abort_flag) {
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
      bars.plan_pool = c.pool;
      bars.plan_off = c.off;
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
  c.pool = bars.plan_pool;
  c.off = bars.plan_off;
  return c;
}

// The epilogue reads the partial output from TMEM two 64-column blocks per round trip.
constexpr int kEpilogueBlocks = 2;

__global__ void __launch_bounds__(kThreads, 1)
attn_main_planned_kernel(const __grid_constant__ TcParams prm) {
#include "attn_main_body.inc"
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
  static std::atomic<bool> attr_set[64];   // per device; setting it twice is harmless
  if (!attr_set[dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(attn_main_planned_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev].store(true, std::memory_order_release);
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

#ifdef MTPATTN_TEST_COVERAGE
#ifndef MTPATTN_COVERAGE_READER
#define MTPATTN_COVERAGE_READER mtpattn_test_coverage_planned
#endif
// Test builds only: copy the first n page counters of this kernel to host memory, then clear
// them (0 or a CUDA error code; -1 for a bad n).
extern "C" int MTPATTN_COVERAGE_READER(uint32_t* host_dst, int64_t n) {
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
