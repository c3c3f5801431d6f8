/*
 * fmha_fp8_varlen.h — C ABI of the fp8 varlen prefill attention in libmtpattn.so (GB300,
 * sm_103a): the second workload of the library, next to the paged verify attention of
 * mtpattn.h.
 *
 * The operation (aiter PR #7375 page, "Summary", "Changes" and the wrapper
 * fmha_fwd_fp8_varlen_asm it describes): packed varlen (THD) e4m3 attention with query/key
 * head dim 192 and value head dim 128.  Sequence b owns query rows cu_seqlens_q[b] ..
 * cu_seqlens_q[b+1]-1 and key/value rows cu_seqlens_k[b] .. cu_seqlens_k[b+1]-1 (Lq and Lk
 * may differ, Lk may be 0).  Query head h reads KV head h / (H_q / H_kv).  The logits are
 * softmax_scale * q_descale * k_descale * <q, k> (per-tensor fp32 descales), the output is
 * v_descale * softmax . v in bf16.  With causal != 0 the mask is bottom-right aligned: query
 * i of a sequence sees keys j <= i + Lk - Lq.  A query that sees no key gets output 0 and
 * log-sum-exp -inf.  The optional log-sum-exp is natural-log, laid out [H_q][total_q] (the
 * varlen layout the page states; the base is our reading).
 *
 * Precision: Q, K and V are the e4m3 inputs themselves (V is widened to f16 inside the
 * kernel, exactly).  The probabilities P (scaled by 2^5 relative to a running row maximum)
 * are rounded once to f16, 11 significant bits, and enter the PV tensor-core product as
 * f16; one e4m3 P would put about 4% of noise on every weight.  Accumulation is fp32.
 *
 * Conventions are those of mtpattn.h: device pointers of the current device, no allocation,
 * no synchronisation, the descales read on the device (graph-capture safe), status codes
 * MTPATTN_* from mtpattn.h, nothing launched on an error return.
 */
#ifndef FMHA_FP8_VARLEN_H
#define FMHA_FP8_VARLEN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FMHA_FP8_HEAD_DIM_QK 192
#define FMHA_FP8_HEAD_DIM_V 128

/* Device-side error bit (OR-ed into the optional status word): a sequence's cu_seqlens
 * entries fall outside [0, total] or decrease, or it has more queries than max_seqlen_q.
 * Its rows are not written. */
#define FMHA_FP8_ERR_CU 32

/*
 *  q             device e4m3 codes [total_q][num_q_heads][192]; byte strides q_stride_tok,
 *                q_stride_head (multiples of 16), unit stride along the head dim, 16-byte
 *                aligned base.
 *  k             device e4m3 [total_k][num_kv_heads][192], strides as for q.
 *  v             device e4m3 [total_k][num_kv_heads][128], strides as for q.
 *  cu_seqlens_q  device int32 [num_seqs + 1], 0 .. total_q, non-decreasing.
 *  cu_seqlens_k  device int32 [num_seqs + 1], 0 .. total_k, non-decreasing.
 *  max_seqlen_q  host int, >= every Lq (sizes the grid; 0 with total_q > 0 is refused with
 *                MTPATTN_E_ARG); max_seqlen_k is accepted for the page's signature and only
 *                checked to be >= 0.
 *  num_q_heads   a multiple of num_kv_heads.
 *  q_descale, k_descale, v_descale   device float32, one element each.
 *  softmax_scale host float (the page's default is 1/sqrt(192); pass it explicitly).
 *  causal        0 or 1 (bottom-right aligned).
 *  out           device bf16 [total_q][num_q_heads][128]; element strides out_stride_tok,
 *                out_stride_head (multiples of 8), unit stride along the head dim.
 *  lse           optional device float32 [num_q_heads][total_q] (NULL = not written).
 *  status        optional device int32; FMHA_FP8_ERR_CU is OR-ed into it, and
 *                MTPATTN_ERR_TIMEOUT if a CTA's pipeline wait ran out (about two seconds
 *                without progress): that CTA's rows and LSEs are then left unwritten.
 *  stream        cudaStream_t as void*.
 * Returns MTPATTN_OK, or MTPATTN_E_ARG / _E_UNSUPPORTED / _E_DEVICE / _E_LAUNCH (see
 * mtpattn.h) before any launch.  One kernel is launched.
 */
int fmha_fwd_fp8_varlen(const void* q, int64_t q_stride_tok, int64_t q_stride_head,
                        const void* k, int64_t k_stride_tok, int64_t k_stride_head,
                        const void* v, int64_t v_stride_tok, int64_t v_stride_head,
                        const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                        int32_t num_seqs, int32_t total_q, int32_t total_k,
                        int32_t max_seqlen_q, int32_t max_seqlen_k,
                        int32_t num_q_heads, int32_t num_kv_heads,
                        const float* q_descale, const float* k_descale, const float* v_descale,
                        float softmax_scale, int32_t causal,
                        void* out, int64_t out_stride_tok, int64_t out_stride_head,
                        float* lse, int32_t* status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FMHA_FP8_VARLEN_H */
