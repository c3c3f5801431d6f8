// Split-KV segment reduce: merge the per-slot partial outputs of one query row
// by their log-sum-exps and round to bf16 (the split-KV segment reduce of the
// aiter PR #5190 page, Modifications).
//
//   M = max_s lse_s,  w_s = 2^(lse_s - M),  out = sum_s w_s o_s / sum_s w_s
//
// Slots with lse = -inf (empty, or no visible key) get weight 0 and their
// partial output is never used, so it need not have been written.  A NaN lse
// marks a row the main kernel flagged as invalid; such rows are written as
// zeros.  The kernel is launched as a programmatic dependent of the main kernel, so
// its CTAs start on the SMs the main kernel's CTAs leave.  Instead of waiting for the
// main grid to complete and flush (griddepcontrol.wait), a CTA waits until the main
// kernel's CTAs have all counted themselves out of the workspace's call counters (each
// after a fence behind its last write), then reads the partials from L2.
//
// Slot pool: when the main kernel laid the partials out unit by unit (AttnParams), a row's
// first LSE slot holds kPoolMarker and the row's first row-slot and piece count; the row's
// warps then load its pool LSEs and walk its slots in blocks of 16 (warp g takes blocks
// g, g + groups, ...).
//
// Work split: the S slots of a row form ceil(S / 16) groups of 16, and each
// (group, half of the row's 256 dims) pair is one warp, 4 dims per lane.  Every
// warp reads all S LSEs (two per lane: the same few cache lines), so each knows M
// and the weight sum; its own group's partial outputs are in flight together, so
// a row costs one round trip of loads whatever S is.  Groups other than the first
// hand their weighted sums to the first through shared memory.
#include "common.cuh"

#include <math.h>

#include <algorithm>

namespace mtpattn {
namespace {

constexpr int kGroup = 16;          // slots per warp
constexpr int kMaxGroups = 8;       // 2 warps each: 512 threads per CTA at most
constexpr long long kCallWaitCycles = 4000000000LL;   // about 2 s: then MTPATTN_ERR_TIMEOUT

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* ptr) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];\n" : "=r"(v) : "l"(ptr) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t ld_relaxed_gpu(const uint32_t* ptr) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];\n" : "=r"(v) : "l"(ptr) : "memory");
  return v;
}

__device__ __forceinline__ float ex2_approx(float x) {   // 2^x, hardware (rel. err ~2^-22)
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

__global__ void __launch_bounds__(512)
attn_reduce_kernel(const AttnParams p, int groups, int rows_per_cta) {
  // Groups 1.. hand their sums to group 0 (one row per CTA): [group - 1][half][lane].  Dynamic
  // shared memory, requested only for S > 16.
  extern __shared__ float4 xfer[];
  __shared__ int s_timed_out;
  // The next kernel on the stream (the next call's main kernel) may start its set-up now;
  // it waits for this grid before it reads or writes anything this grid touches.
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  // This grid started only after every main-kernel CTA had counted itself in, so `started`
  // is the main grid's CTA count; wait (bounded) until all of them have counted out.
  if (threadIdx.x == 0) {
    const uint32_t started = ld_relaxed_gpu(p.call_ctr);
    bool ok = ld_acquire_gpu(p.call_ctr + 1) == started;
    if (!ok) {
      const long long t0 = clock64();
      while (!(ok = ld_acquire_gpu(p.call_ctr + 1) == started) && clock64() - t0 < kCallWaitCycles) {
      }
    }
    s_timed_out = !ok;
    if (!ok) set_status(p.status, MTPATTN_ERR_TIMEOUT);
  }
  __syncthreads();
  // Every main-kernel CTA is done with its tiles: put the tile counters back to zero for the
  // next call (which waits for this grid before it claims any).
  if (blockIdx.x == 0) {
    const int units = min(p.num_seqs * p.num_kv_heads, kMaxTileCounters);
    for (int i = threadIdx.x; i < units; i += blockDim.x) p.tile_ctr[i] = 0u;
  }
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int wpr = 2 * groups;                      // warps per row
  const int g = (warp % wpr) >> 1;                 // slot group of this warp
  const int part = warp & 1;                       // half of the row's dims
  const int64_t row = static_cast<int64_t>(blockIdx.x) * rows_per_cta + warp / wpr;
  const int64_t rows = static_cast<int64_t>(p.total_q) * p.num_q_heads;
  const bool live = row < rows;
  const int S = p.num_segments;
  const int s_lo = g * kGroup;
  // Slots below slots_used are the ones most rows use: their partial outputs are loaded
  // together with the LSEs.  Others of the group only where their weight is not 0.  A slot
  // of weight 0 may hold anything, so its values are dropped by a select, never multiplied.
  const int n_spec = live ? max(0, min(min(p.slots_used, S) - s_lo, kGroup)) : 0;
  const float* lse = p.lse_part + (live ? row : 0) * S;
  // (loads through L2 only: no line of this call's partials may come from L1)
  const float l0 = live && lane < S ? __ldcg(lse + lane) : -INFINITY;
  const float l1 = live && lane + 32 < S ? __ldcg(lse + lane + 32) : -INFINITY;
  const float* ob = p.o_part + (live ? row : 0) * S * kHeadDim + part * 128 + lane * 4;
  float4 a[kGroup];
#pragma unroll
  for (int i = 0; i < kGroup; ++i)
    if (i < n_spec) a[i] = __ldcg(reinterpret_cast<const float4*>(ob + static_cast<int64_t>(s_lo + i) * kHeadDim));
  // The row's slots: P of them, LSEs lv[k] of slots lane + 32 k on each lane, partial outputs
  // from `ob`.  Slot pool (see AttnParams): the first LSE slot redirects to the row's partials
  // (honoured only if this call allowed the pool, and only inside this call's pool; otherwise
  // the row is treated as an error), which costs one more round trip; the loads above were
  // speculative.
  float lv[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) lv[k] = k == 0 ? l0 : (k == 1 ? l1 : -INFINITY);
  int P = S;
  int bad = s_timed_out;                           // then the partials are unknown: zeros
  bool spec = true;
  if (live && p.slot_pool && __shfl_sync(0xffffffffu, __float_as_uint(l0), 0) == kPoolMarker) {
    const int off = __shfl_sync(0xffffffffu, __float_as_int(l0), 1);
    P = __shfl_sync(0xffffffffu, __float_as_int(l0), 2);
    spec = false;
    if (off < 0 || P < 1 || P > 256 || off > p.pool_cap - P) {
      bad = 1;
      P = 0;
    } else {
      const float* pl = p.pool_lse + off;
#pragma unroll
      for (int k = 0; k < 8; ++k) lv[k] = lane + 32 * k < P ? __ldcg(pl + lane + 32 * k) : -INFINITY;
      ob = p.o_part + static_cast<int64_t>(off) * kHeadDim + part * 128 + lane * 4;
    }
  }
  float mx = -INFINITY;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    bad |= isnan(lv[k]);
    mx = fmaxf(mx, lv[k]);
  }
#pragma unroll
  for (int off2 = 16; off2 > 0; off2 >>= 1) {
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off2));
    bad |= __shfl_xor_sync(0xffffffffu, bad, off2);
  }
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f;
  if (!bad && mx != -INFINITY) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      lv[k] = lv[k] == -INFINITY ? 0.f : ex2_approx(lv[k] - mx);   // now the weights
      wsum += lv[k];
    }
#pragma unroll
    for (int off2 = 16; off2 > 0; off2 >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, off2);
    // This warp's blocks of 16 slots: g, g + groups, ... (each inside one lane group of 32).
    // All the weights of a block first, then every load of the block at once.
#pragma unroll 1
    for (int s0 = s_lo; s0 < P; s0 += groups * kGroup) {
      const int kk = s0 >> 5;
      float src = lv[0];
#pragma unroll
      for (int k = 1; k < 8; ++k)
        if (k == kk) src = lv[k];
      float w[kGroup];
#pragma unroll
      for (int i = 0; i < kGroup; ++i) w[i] = __shfl_sync(0xffffffffu, src, (s0 & 31) + i);
      const int have = spec && s0 == s_lo ? n_spec : 0;     // already in flight
#pragma unroll
      for (int i = 0; i < kGroup; ++i)
        if (i >= have && s0 + i < P && w[i] != 0.f)          // uniform across the warp
          a[i] = __ldcg(reinterpret_cast<const float4*>(ob + static_cast<int64_t>(s0 + i) * kHeadDim));
      // A slot of weight 0 may hold anything: its values are dropped by a select.
#pragma unroll
      for (int i = 0; i < kGroup; ++i) {
        if (s0 + i < P && w[i] != 0.f) {
          acc.x = fmaf(w[i], a[i].x, acc.x); acc.y = fmaf(w[i], a[i].y, acc.y);
          acc.z = fmaf(w[i], a[i].z, acc.z); acc.w = fmaf(w[i], a[i].w, acc.w);
        }
      }
    }
  }
  if (groups > 1) {                                 // one row per CTA
    if (g > 0) xfer[((g - 1) * 2 + part) * 32 + lane] = acc;
    __syncthreads();
    if (g > 0) return;
    for (int h = 1; h < groups; ++h) {
      const float4 v = xfer[((h - 1) * 2 + part) * 32 + lane];
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
  }
  if (!live || g > 0) return;
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  const int64_t tok = row / p.num_q_heads, head = row - tok * p.num_q_heads;
  __nv_bfloat16* dst = p.out + tok * p.out_stride_tok + head * p.out_stride_head + part * 128 + lane * 4;
  const __nv_bfloat162 v0 = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
  const __nv_bfloat162 v1 = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
  *reinterpret_cast<uint2*>(dst) = make_uint2(*reinterpret_cast<const uint32_t*>(&v0),
                                              *reinterpret_cast<const uint32_t*>(&v1));
}

}  // namespace

cudaError_t launch_attn_reduce(const AttnParams& p, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(p.total_q) * p.num_q_heads;
  int groups = (p.num_segments + kGroup - 1) / kGroup;
  // With the slot pool a row may have up to one slot per SM: more groups per row let such a
  // row load its slots in fewer rounds (the row-major rows leave the extra warps idle), as long
  // as the whole grid stays one wave: a CTA of g groups holds 1/g of an SM's registers at
  // 128 per thread (8 groups, 512 threads, at most).
  if (p.slot_pool && rows > 0) {
    const int sms = device_sm_count(-1);
    if (sms > 0) {
      const int64_t fit = static_cast<int64_t>(kMaxGroups) * sms / rows;   // groups for one wave
      const int want = std::min<int64_t>(kMaxGroups, std::min<int64_t>(fit, (sms + kGroup - 1) / kGroup));
      groups = std::max(groups, want);
    }
  }
  const int rows_per_cta = groups == 1 ? 2 : 1;    // 128 threads for S <= 16, else 64 per group
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((rows + rows_per_cta - 1) / rows_per_cta));
  cfg.blockDim = dim3(rows_per_cta * 2 * groups * 32);
  cfg.dynamicSmemBytes = static_cast<size_t>(groups - 1) * 2 * 32 * sizeof(float4);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, attn_reduce_kernel, p, groups, rows_per_cta);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace mtpattn
