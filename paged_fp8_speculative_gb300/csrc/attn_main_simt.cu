// Split-KV main kernel, CUDA-core version (float32 arithmetic throughout).
//
// One CTA per (segment s, sequence b, KV head h) — the decomposition of the
// aiter PR #5190 page (Modifications: grid = segments x sequences x kv heads).
// The CTA packs the q_len x ratio query rows of its KV head (GQA packing, same
// page: "supports GQA ratios 16 and 8 natively"), streams its segment's pages
// of K and V straight from the paged NHD cache through the block table with
// 16-byte cp.async copies into a two-stage shared-memory ring, and runs an
// online softmax (running max m, running sum l, rescale by 2^(m_old - m_new))
// over the pages.  It writes the segment's normalised partial output and its
// log2-sum-exp2; empty segments write o = 0, lse = -inf.
#include "common.cuh"

#include <cuda_fp8.h>
#include <math.h>

namespace mtpattn {
namespace {

constexpr int kThreads = 256;
constexpr int kQStride = kHeadDim + 4;          // floats per Q row in smem (bank spread)
constexpr int kKStride = kHeadDim + 16;         // bytes per K row in smem (bank spread)
constexpr int kSStride = kPage + 1;             // floats per score row

struct __align__(16) Smem {
  float q[kMaxRows * kQStride];                 // 66,560 B
  uint8_t k[2][kPage * kKStride];               //  8,704 B
  uint8_t v[2][kPage * kHeadDim];               //  8,192 B
  float s[kMaxRows * kSStride];                 //  4,352 B
  float m[kMaxRows], l[kMaxRows], alpha[kMaxRows];
  int32_t phys[2];
};

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n"); }

// Four e4m3 codes -> four floats (exact: every e4m3 value is an f16 value).
__device__ __forceinline__ void e4m3x4_to_float(uint32_t w, float* f) {
  __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w & 0xFFFF), __NV_E4M3);
  __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w >> 16), __NV_E4M3);
  float2 a = __half22float2(*reinterpret_cast<__half2*>(&lo));
  float2 b = __half22float2(*reinterpret_cast<__half2*>(&hi));
  f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
}

// Issue the 16-byte copies of one page of K and V (head h) into ring slot `buf`.
__device__ __forceinline__ void load_page(Smem& sm, const AttnParams& p, int32_t phys, int h,
                                          int buf, int tid) {
  const int slot = tid >> 4;            // 16 keys
  const int chunk = tid & 15;           // 16 chunks of 16 B per 256-B key row
  const size_t row = (static_cast<size_t>(phys) * kPage + slot) * p.num_kv_heads + h;
  cp_async16(&sm.k[buf][slot * kKStride + chunk * 16], p.k_cache + row * kHeadDim + chunk * 16);
  cp_async16(&sm.v[buf][slot * kHeadDim + chunk * 16], p.v_cache + row * kHeadDim + chunk * 16);
}

__global__ void __launch_bounds__(kThreads)
attn_main_simt_kernel(const AttnParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
  const int tid = threadIdx.x;
  const int s = blockIdx.x, b = blockIdx.y, h = blockIdx.z;
  const int S = p.num_segments;

  const int L = p.seq_lens[b];
  const int q0 = p.cu_q[b];
  const int q1 = p.cu_q[b + 1];
  const int ql = q1 - q0;
  const bool rows_known = q0 >= 0 && q1 <= p.total_q && ql >= 1 && ql <= kMaxQLen;
  int err = 0;
  if (!rows_known) err |= MTPATTN_ERR_QLEN;
  else if (ql > L) err |= MTPATTN_ERR_QLEN_GT_SEQ;
  const int n_pages = (L + kPage - 1) / kPage;
  if (!err && n_pages > p.max_pages) err |= MTPATTN_ERR_SEQ_TOO_LONG;
  const int R = rows_known ? ql * p.ratio : 0;

  int pb = 0, pe = 0;
  if (!err) segment_pages(n_pages, S, s, &pb, &pe);
  const int32_t* bt = p.block_tables + static_cast<size_t>(b) * p.max_pages;

  // Row r = t * ratio + g  <->  query token q0 + t, query head h * ratio + g.
  auto out_row = [&](int r) -> int64_t {
    const int t = r / p.ratio, g = r - t * p.ratio;
    return static_cast<int64_t>(q0 + t) * p.num_q_heads + h * p.ratio + g;
  };

  // Validate every block-table entry of the segment before touching the cache.
  if (!err) {
    int bad = 0;
    for (int i = pb + tid; i < pe; i += kThreads) {
      const int32_t e = bt[i];
      bad |= (e < 0 || e >= p.num_pages);
    }
    if (__syncthreads_or(bad)) err |= MTPATTN_ERR_PAGE;
  }
  if (err) {
    if (tid == 0) set_status(p.status, err);
    // Rows that can be identified get a NaN LSE: the reduce writes them as zeros.
    for (int r = tid; r < R; r += kThreads) p.lse_part[out_row(r) * S + s] = __int_as_float(0x7fc00000);
    return;
  }

  if (pb >= pe) {  // empty segment: neutral partials
    for (int i = tid; i < R * kHeadDim; i += kThreads) {
      const int r = i / kHeadDim, d = i - r * kHeadDim;
      p.o_part[(out_row(r) * S + s) * kHeadDim + d] = 0.f;
    }
    for (int r = tid; r < R; r += kThreads) p.lse_part[out_row(r) * S + s] = -INFINITY;
    return;
  }

  // Kick off the first page, then stage Q (bf16 -> float32) while it flies.
  if (tid == 0) sm.phys[0] = bt[pb];
  __syncthreads();
  load_page(sm, p, sm.phys[0], h, 0, tid);
  cp_async_commit();
  for (int i = tid; i < kMaxRows * (kHeadDim / 8); i += kThreads) {
    const int r = i / (kHeadDim / 8), c = (i - r * (kHeadDim / 8)) * 8;
    float* dst = &sm.q[r * kQStride + c];
    if (r < R) {
      const int t = r / p.ratio, g = r - t * p.ratio;
      const __nv_bfloat16* src = p.q + static_cast<int64_t>(q0 + t) * p.q_stride_tok +
                                 static_cast<int64_t>(h * p.ratio + g) * p.q_stride_head + c;
      const uint4 raw = *reinterpret_cast<const uint4*>(src);
      const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        dst[2 * j] = __uint_as_float(w[j] << 16);
        dst[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) dst[j] = 0.f;
    }
  }
  if (tid < kMaxRows) { sm.m[tid] = -INFINITY; sm.l[tid] = 0.f; }

  const float qk_scale = p.scale_log2 * __ldg(p.k_descale);
  // PV ownership: 4 consecutive dims x 16 rows per thread.
  const int dq = tid & 63, rq = tid >> 6;
  float acc[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

  // QK ownership: one key x 4 rows per thread.
  const int kk = tid & 15, rg = tid >> 4;

  for (int pg = pb; pg < pe; ++pg) {
    const int buf = (pg - pb) & 1;
    cp_async_wait_all();
    __syncthreads();                                   // page pg landed; ring slot buf^1 free
    if (pg + 1 < pe) {
      const int32_t nxt = bt[pg + 1];
      load_page(sm, p, nxt, h, buf ^ 1, tid);
      cp_async_commit();
    }

    // ---- S = Q K^T for 4 rows x 1 key -----------------------------------------------------
    {
      float dot[4] = {0.f, 0.f, 0.f, 0.f};
      const uint8_t* krow = &sm.k[buf][kk * kKStride];
#pragma unroll 4
      for (int d = 0; d < kHeadDim; d += 16) {
        const uint4 kw = *reinterpret_cast<const uint4*>(krow + d);
        float kf[16];
        e4m3x4_to_float(kw.x, kf);
        e4m3x4_to_float(kw.y, kf + 4);
        e4m3x4_to_float(kw.z, kf + 8);
        e4m3x4_to_float(kw.w, kf + 12);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const float* qr = &sm.q[(rg * 4 + r) * kQStride + d];
#pragma unroll
          for (int j = 0; j < 16; j += 4) {
            const float4 qv = *reinterpret_cast<const float4*>(qr + j);
            dot[r] = fmaf(qv.x, kf[j], dot[r]);
            dot[r] = fmaf(qv.y, kf[j + 1], dot[r]);
            dot[r] = fmaf(qv.z, kf[j + 2], dot[r]);
            dot[r] = fmaf(qv.w, kf[j + 3], dot[r]);
          }
        }
      }
      const int key = pg * kPage + kk;
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int row = rg * 4 + r;
        const int t = row / p.ratio;
        const bool vis = row < R && key <= L - ql + t;
        sm.s[row * kSStride + kk] = vis ? dot[r] * qk_scale : -INFINITY;
      }
    }
    __syncthreads();

    // ---- online softmax, one thread per row ------------------------------------------------
    if (tid < kMaxRows) {
      float* srow = &sm.s[tid * kSStride];
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < kPage; ++j) mx = fmaxf(mx, srow[j]);
      const float m_old = sm.m[tid];
      const float m_new = fmaxf(m_old, mx);
      float alpha = 1.f, sum = 0.f;
      if (m_new == -INFINITY) {
#pragma unroll
        for (int j = 0; j < kPage; ++j) srow[j] = 0.f;
      } else {
        alpha = exp2f(m_old - m_new);                  // 0 when m_old = -inf
#pragma unroll
        for (int j = 0; j < kPage; ++j) {
          const float pj = exp2f(srow[j] - m_new);
          srow[j] = pj;
          sum += pj;
        }
      }
      sm.l[tid] = sm.l[tid] * alpha + sum;
      sm.m[tid] = m_new;
      sm.alpha[tid] = alpha;
    }
    __syncthreads();

    // ---- O = alpha O + P V -----------------------------------------------------------------
    {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float a = sm.alpha[rq * 16 + i];
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] *= a;
      }
      const uint8_t* vb = sm.v[buf];
#pragma unroll 4
      for (int j = 0; j < kPage; ++j) {
        float vf[4];
        e4m3x4_to_float(*reinterpret_cast<const uint32_t*>(vb + j * kHeadDim + dq * 4), vf);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float pij = sm.s[(rq * 16 + i) * kSStride + j];
          acc[i][0] = fmaf(pij, vf[0], acc[i][0]);
          acc[i][1] = fmaf(pij, vf[1], acc[i][1]);
          acc[i][2] = fmaf(pij, vf[2], acc[i][2]);
          acc[i][3] = fmaf(pij, vf[3], acc[i][3]);
        }
      }
    }
  }

  // ---- epilogue: o_s = v_descale * acc / l, lse_s = m + log2 l ----------------------------
  __syncthreads();
  const float vd = __ldg(p.v_descale);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int r = rq * 16 + i;
    if (r >= R) continue;
    const float l = sm.l[r];
    const float inv = l > 0.f ? vd / l : 0.f;
    float4 o = make_float4(acc[i][0] * inv, acc[i][1] * inv, acc[i][2] * inv, acc[i][3] * inv);
    *reinterpret_cast<float4*>(&p.o_part[(out_row(r) * S + s) * kHeadDim + dq * 4]) = o;
  }
  if (tid < R) {
    const float l = sm.l[tid];
    p.lse_part[out_row(tid) * S + s] = l > 0.f ? sm.m[tid] + log2f(l) : -INFINITY;
  }
}

}  // namespace

cudaError_t launch_attn_main_simt(const AttnParams& p, cudaStream_t stream) {
  const size_t smem = sizeof(Smem);
  cudaError_t e = cudaFuncSetAttribute(attn_main_simt_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid(p.num_segments, p.num_seqs, p.num_kv_heads);
  attn_main_simt_kernel<<<grid, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mtpattn
