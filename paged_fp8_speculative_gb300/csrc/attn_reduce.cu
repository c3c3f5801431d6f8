// Split-KV segment reduce: merge the per-slot partial outputs of one query row
// by their log-sum-exps and round to bf16 (the split-KV segment reduce of the
// aiter PR #5190 page, Modifications).
//
//   M = max_s lse_s,  w_s = 2^(lse_s - M),  out = sum_s w_s o_s / sum_s w_s
//
// Slots with lse = -inf (empty, or no visible key) get weight 0 and their
// partial output is never used, so it need not have been written.  Only the
// slots the main kernel's chunking can reach (slots_used) are read.  A NaN lse
// marks a row the main kernel flagged as invalid; such rows are written as
// zeros.  Two warps per row, 4 dims per lane; the loads of up to 16 slots are in
// flight together.  The kernel is launched as a programmatic dependent of the main
// kernel: it may start while the main kernel drains and waits (griddepcontrol)
// until the main kernel's results are visible.
#include "common.cuh"

#include <math.h>

namespace mtpattn {
namespace {

constexpr int kWarpsPerCta = 4;
constexpr int kWarpsPerRow = 2;     // each warp merges 128 of the row's 256 dims, 4 per lane
constexpr int kGroup = 16;          // slots whose loads are in flight together

__global__ void __launch_bounds__(kWarpsPerCta * 32)
attn_reduce_kernel(const AttnParams p) {
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  // The next kernel on the stream (the next call's main kernel) may start its set-up now;
  // it waits for this grid before it reads or writes anything this grid touches.
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  // The main kernel is complete: put its tile counters back to zero for the next call.
  if (blockIdx.x == 0) {
    const int units = min(p.num_seqs * p.num_kv_heads, kMaxTileCounters);
    for (int i = threadIdx.x; i < units; i += blockDim.x) p.tile_ctr[i] = 0u;
  }
  const int lane = threadIdx.x & 31;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * kWarpsPerCta + (threadIdx.x >> 5);
  const int64_t row = gw / kWarpsPerRow;
  const int part = static_cast<int>(gw % kWarpsPerRow);
  const int64_t rows = static_cast<int64_t>(p.total_q) * p.num_q_heads;
  if (row >= rows) return;
  const int S = p.num_segments;
  const int n = p.slots_used;                // slots at or beyond n were never written
  const float* lse = p.lse_part + row * S;
  const float* o = p.o_part + row * S * kHeadDim + part * 128 + lane * 4;

  // Each lane holds slots lane and lane + 32.  The partial outputs of the first group are
  // loaded together with the LSEs (one round trip); a slot whose weight turns out to be 0
  // may hold anything, so its values are dropped by a select, never multiplied.
  const float l0 = lane < n ? lse[lane] : -INFINITY;
  const float l1 = lane + 32 < n ? lse[lane + 32] : -INFINITY;
  float4 a[kGroup];
#pragma unroll
  for (int g = 0; g < kGroup; ++g)
    if (g < n) a[g] = *reinterpret_cast<const float4*>(o + static_cast<int64_t>(g) * kHeadDim);
  int bad = isnan(l0) || isnan(l1);
  float mx = fmaxf(l0, l1);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    bad |= __shfl_xor_sync(0xffffffffu, bad, off);
  }
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f;
  if (!bad && mx != -INFINITY) {
    const float w0 = l0 == -INFINITY ? 0.f : exp2f(l0 - mx);
    const float w1 = l1 == -INFINITY ? 0.f : exp2f(l1 - mx);
    for (int s0 = 0; s0 < n; s0 += kGroup) {
      if (s0 > 0) {
#pragma unroll
        for (int g = 0; g < kGroup; ++g)
          if (s0 + g < n) a[g] = *reinterpret_cast<const float4*>(o + static_cast<int64_t>(s0 + g) * kHeadDim);
      }
#pragma unroll
      for (int g = 0; g < kGroup; ++g) {
        const int s2 = s0 + g;
        const float w = __shfl_sync(0xffffffffu, s2 < 32 ? w0 : w1, s2 & 31);
        if (s2 < n && w != 0.f) {                // uniform across the warp (one row)
          wsum += w;
          acc.x = fmaf(w, a[g].x, acc.x); acc.y = fmaf(w, a[g].y, acc.y);
          acc.z = fmaf(w, a[g].z, acc.z); acc.w = fmaf(w, a[g].w, acc.w);
        }
      }
    }
  }
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
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((rows * kWarpsPerRow + kWarpsPerCta - 1) / kWarpsPerCta));
  cfg.blockDim = dim3(kWarpsPerCta * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, attn_reduce_kernel, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace mtpattn
