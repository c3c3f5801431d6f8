/*
 * mtpattn.h — C ABI of the paged fp8 split-KV attention library (libmtpattn.so)
 * for the speculative-decoding verify, draft-extend and decode steps on GB300 (sm_103a).
 *
 * The operation.  Each sequence b has q_len_b query tokens (1..4, bf16,
 * head_dim 256) packed at rows cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 of q, and
 * seq_lens[b] keys in a paged NHD page-16 fp8 e4m3 K/V cache read in place
 * through block_tables.  Query token t sees keys 0 .. seq_lens[b]-q_len_b+t
 * (causal over the last q_len positions, bottom-right aligned); query head j
 * reads KV head j / ratio with ratio = H_q / H_kv in {8, 16}; logits are
 * softmax_scale * k_descale * <q, K>, the output is v_descale * softmax · V,
 * rounded to bf16.  Sources: aiter PR #5190 page ("gfx950 assembly MTP-verify
 * attention for head_dim 256 fp8 paged KV", Motivation, Modifications, Kernel
 * notes, Supported) and SGLang PR #37465 page ("gfx950 assembly attention for
 * EAGLE verify, draft extend and decode", Modifications: q_len 1..4 handled in
 * one kernel for verify, draft extend and decode).  seq_lens counts the current
 * query tokens (their K/V are already in the cache).
 *
 * Split-KV: the keys of each (sequence, KV head) are cut into pieces of whole
 * pages; a main kernel writes one partial output and one log-sum-exp per (row,
 * piece) into the caller's workspace and a second kernel merges them by their
 * LSE into the bf16 output (aiter PR #5190 page, Modifications: the split-KV
 * main kernel and its segment reduce).  num_segments (S) is the number of split
 * slots per (sequence, KV head): the pages of all units are shared out in equal
 * chunks over the SMs, no unit is cut into more than S pieces (unless S was left to
 * the library, see num_segments below), and slots a unit does not use are written empty.  Any S in [1, 64] gives the same result up to
 * float32 re-association; S = 1 keeps every unit whole.
 *
 * Balanced scheduling (the default): when every unit is cut into whole pieces
 * and each SM holds one piece, the pieces of a unit share its 128-key tiles
 * through a counter in the workspace, so SMs that stream faster take more
 * tiles.  Which piece sums which tiles then varies from call to call: results
 * agree to float32 re-association, not bit for bit.  After
 * mtp_verify_attn_set_deterministic(1) every piece keeps a fixed page range and
 * repeated calls are bit-identical.
 *
 * Conventions for every entry point:
 *  - Pointers marked "device" must be CUDA device memory of the current device;
 *    the library never dereferences them on the host, never allocates, never
 *    synchronises and never copies device data to the host in mtp_verify_attn_fwd,
 *    so a call may be captured in a CUDA graph.  The descales are read on the
 *    device for the same reason (aiter PR #5190 page, Kernel notes).
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *  - The caller owns every buffer.  The library keeps only host-side caches: the
 *    SM count and each kernel's shared-memory attribute per device, and the TMA
 *    tensor maps of the last few K/V caches (keyed by address and shape), all safe
 *    to use from several host threads at once; plus the static device array of
 *    mtp_verify_attn_fwd_static_scratch.
 *  - Return codes: MTPATTN_OK or a negative MTPATTN_E_*.  On an error return
 *    nothing was launched.  Nothing prints, throws or traps.
 */
#ifndef MTPATTN_H
#define MTPATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MTPATTN_OK 0
#define MTPATTN_E_ARG (-1)          /* null pointer, negative count, bad stride or alignment */
#define MTPATTN_E_UNSUPPORTED (-2)  /* outside the envelope: head_dim, page size, ratio, segments */
#define MTPATTN_E_DEVICE (-3)       /* a pointer is not device memory of the current device, or no device */
#define MTPATTN_E_WORKSPACE (-4)    /* workspace null, too small or not 256-byte aligned */
#define MTPATTN_E_LAUNCH (-5)       /* a kernel launch failed (cudaGetLastError after launch) */
#define MTPATTN_E_SCRATCH_LIMIT (-6) /* the call needs more than MTPATTN_STATIC_SCRATCH_BYTES of scratch */

/* Device-side error bits OR-ed into the optional `status` word (device int32).
 * The affected rows are written as zeros; nothing outside the given buffers is read. */
#define MTPATTN_ERR_QLEN 1          /* q_len_b outside [1, 4] or cu_seqlens_q not ascending within total_q */
#define MTPATTN_ERR_QLEN_GT_SEQ 2   /* q_len_b > seq_lens[b] */
#define MTPATTN_ERR_PAGE 4          /* a block-table entry needed for a key is outside [0, num_pages) */
#define MTPATTN_ERR_SEQ_TOO_LONG 8  /* seq_lens[b] > 16 * max_pages_per_seq */
#define MTPATTN_ERR_TIMEOUT 16      /* a pipeline wait inside the main kernel gave up (about 2 s
                                       without progress); that call's output is not valid */

#define MTPATTN_HEAD_DIM 256
#define MTPATTN_PAGE_SIZE 16
#define MTPATTN_MAX_SEGMENTS 64
#define MTPATTN_MAX_Q_LEN 4

/*
 * Number of split slots S per (sequence, KV head) for a batch shape, in [1, 64]
 * (aiter PR #5190 page, Modifications: mtp_verify_attn_num_segments(); no
 * formula is printed).  Our rule depends on the scheduling switch below:
 *  - planned scheduling (and U = num_seqs * num_kv_heads <= 256 and <= SMs):
 *    S = min(SMs - U + 1, ceil(max_pages_per_seq / 8)), clamped to [1, 64]: the
 *    pieces are sized from the lengths on the device, and S only caps how many
 *    SMs one long sequence may take;
 *  - otherwise: the page share of one SM is
 *    ceil(num_seqs * num_kv_heads * max_pages_per_seq / SMs), and S is the number
 *    of shares a full-length unit can touch, ceil(max_pages_per_seq / share) + 1,
 *    capped at 64.
 * device < 0 means the current device.  Returns a negative MTPATTN_E_* on bad
 * arguments or when the device cannot be queried.
 */
int32_t mtp_verify_attn_num_segments(int32_t num_seqs, int32_t num_kv_heads,
                                     int32_t max_pages_per_seq, int32_t device);

/*
 * Bytes of device workspace mtp_verify_attn_fwd needs (the library's own sizing
 * rule; the pages print no counterpart): a header of MTPATTN_WORKSPACE_HEADER_BYTES
 * (4096 bytes of tile counters, one per (sequence, KV head) unit up to 1024 units,
 * then two 32-bit call counters: the main kernel's CTAs count themselves in when
 * they start and out after their last write, and the reduce merges once the two
 * agree), then float32 partial log-sum-exps [total_q * num_q_heads][num_segments],
 * then float32 partial outputs [total_q * num_q_heads][num_segments][256], each
 * region 256-byte aligned.  Returns 0 for invalid arguments.
 */
#define MTPATTN_WORKSPACE_HEADER_BYTES 4352

size_t mtp_verify_attn_workspace_size(int32_t total_q, int32_t num_q_heads, int32_t num_segments);

/*
 * out = paged fp8 verify / draft-extend / decode attention (see the top of this file).
 *
 *  q            device bf16 [total_q][num_q_heads][256]; element strides q_stride_tok,
 *               q_stride_head (multiples of 8), unit stride along head_dim; 16-byte aligned.
 *  k_cache,     device e4m3 codes [num_pages][16][num_kv_heads][256], contiguous,
 *  v_cache      16-byte aligned (NHD pages, read in place).
 *  block_tables device int32 [num_seqs][max_pages_per_seq]; entries past
 *               ceil(seq_lens[b]/16) are never read.
 *  seq_lens     device int32 [num_seqs], keys per sequence including the query tokens.
 *  cu_seqlens_q device int32 [num_seqs+1], cu[0] = 0, cu[num_seqs] = total_q, 1 <= q_len <= 4.
 *  num_q_heads  = ratio * num_kv_heads with ratio 8 or 16.
 *  k_descale,   device float32, one element each (per-tensor descales).
 *  v_descale
 *  softmax_scale  host float, multiplies the logits (usually 1/sqrt(256)).
 *  num_segments in [1, 64], or 0 for mtp_verify_attn_num_segments().  With 0 (and S >= 3,
 *               planned scheduling) the workspace's total_q * num_q_heads * S partial slots
 *               are shared out by length: a long sequence may take more than S pieces (at
 *               most one per SM) when short ones use fewer.  A ragged batch with one long
 *               sequence then streams it on every SM instead of on S of them.
 *  workspace    device, >= mtp_verify_attn_workspace_size(...) bytes, 256-byte aligned.
 *               Its first MTPATTN_WORKSPACE_HEADER_BYTES bytes (the counter header) must
 *               be zero before the workspace's first use (e.g. one cudaMemset); every
 *               call that returns MTPATTN_OK, also one that reports a device error,
 *               leaves the tile counters zero and the two call counters equal, so the
 *               workspace can be reused by calls of any shape without clearing.  After
 *               MTPATTN_E_LAUNCH the main kernel may have run without the reduce that
 *               resets the tile counters: zero the header again before reusing it.
 *               The rest need not be initialised.  Calls that overlap on the GPU must
 *               use different workspaces.
 *  out          device bf16 [total_q][num_q_heads][256]; element strides out_stride_tok,
 *               out_stride_head (multiples of 8), unit stride along head_dim.
 *  status       optional device int32 (NULL = none); device-side MTPATTN_ERR_* bits are
 *               OR-ed into it and never cleared by the library.
 *  stream       cudaStream_t as void*.
 * Two kernels are launched on `stream`: the split-KV main kernel and the segment reduce.
 */
int mtp_verify_attn_fwd(const void* q, int64_t q_stride_tok, int64_t q_stride_head,
                        const void* k_cache, const void* v_cache, int64_t num_pages,
                        const int32_t* block_tables, int32_t max_pages_per_seq,
                        const int32_t* seq_lens, const int32_t* cu_seqlens_q,
                        int32_t num_seqs, int32_t total_q, int32_t num_q_heads,
                        int32_t num_kv_heads, const float* k_descale, const float* v_descale,
                        float softmax_scale, int32_t num_segments,
                        void* workspace, size_t workspace_bytes,
                        void* out, int64_t out_stride_tok, int64_t out_stride_head,
                        int32_t* status, void* stream);

/*
 * The same operation in the pages' precision class (aiter PR #5190 page, "Kernel notes":
 * "Q and P are quantized to fp8"; its "Microbenchmark" notes give 0.13 sigma as that
 * quantisation's error floor).  Arguments, workspace rules, return codes and status bits
 * are those of mtp_verify_attn_fwd; what differs:
 *  - each query row is scaled by a power of two (its largest |q| to [128, 256)) and rounded
 *    once to e4m3, and each probability p * 2^(8 - 3) (at most 256) is rounded once to e4m3
 *    before PV, instead of being carried as two e4m3 terms; the result differs from the
 *    exact attention by up to about 0.15 of the output's standard deviation on data whose
 *    logits are O(1), against about 0.01 for mtp_verify_attn_fwd;
 *  - it always uses planned scheduling, whatever mtp_verify_attn_set_scheduling chose, and
 *    returns MTPATTN_E_UNSUPPORTED (launching nothing) for batches planned scheduling does
 *    not take: more (sequence, KV head) units than 256 or than the GPU's SMs.
 * The two tiers run at the same speed here (the K/V stream bounds both); this one exists
 * for callers that want the pages' numerics.
 */
int mtp_verify_attn_fwd_qp_fp8(const void* q, int64_t q_stride_tok, int64_t q_stride_head,
                               const void* k_cache, const void* v_cache, int64_t num_pages,
                               const int32_t* block_tables, int32_t max_pages_per_seq,
                               const int32_t* seq_lens, const int32_t* cu_seqlens_q,
                               int32_t num_seqs, int32_t total_q, int32_t num_q_heads,
                               int32_t num_kv_heads, const float* k_descale,
                               const float* v_descale, float softmax_scale,
                               int32_t num_segments, void* workspace, size_t workspace_bytes,
                               void* out, int64_t out_stride_tok, int64_t out_stride_head,
                               int32_t* status, void* stream);

/*
 * Size of the library-owned device scratch array used by
 * mtp_verify_attn_fwd_static_scratch: 32 MiB, held on every GPU that loads the
 * library until the process exits.
 */
#define MTPATTN_STATIC_SCRATCH_BYTES (32u << 20)

/*
 * mtp_verify_attn_fwd without a caller workspace, for callers that cannot
 * allocate device memory: code inside another framework's memory pool that may
 * not call cudaMalloc, launches issued while a CUDA graph is being captured
 * (a fresh cudaMalloc is not allowed there), or latency-critical loops that
 * must not reach cudaMalloc / cudaFree because those can synchronise the device.
 * The pages have no counterpart of this entry point.
 *
 * Arguments are those of mtp_verify_attn_fwd minus workspace / workspace_bytes;
 * the caller still passes every input and the output.  The split-KV partials go
 * to a file-scope device array of MTPATTN_STATIC_SCRATCH_BYTES that the library
 * owns; it allocates nothing (no cudaMalloc, cudaFree or allocating library call).
 * Calls needing more scratch than that (mtp_verify_attn_workspace_size() of the
 * resolved segment count) return MTPATTN_E_SCRATCH_LIMIT and launch nothing.
 * The first call on each device looks up the array's device address with that
 * device current (cudaGetSymbolAddress), caches it, and clears the array's
 * counter header (MTPATTN_WORKSPACE_HEADER_BYTES) with cudaMemsetAsync on `stream`, so the clear is
 * ordered before the call's kernels on any kind of stream; make that first call
 * before any stream capture.  After a call that returned MTPATTN_E_LAUNCH (its
 * reduce may not have run to reset the counters) the next call clears the
 * header again the same way.
 * Every call on a device shares the one array and leaves its contents behind,
 * so calls that overlap on the GPU (other streams, other threads) race on it and
 * must be serialised by the caller.  Host calls are serialised by a mutex.
 * Other return codes and the device status bits are those of mtp_verify_attn_fwd.
 */
int mtp_verify_attn_fwd_static_scratch(const void* q, int64_t q_stride_tok, int64_t q_stride_head,
                                       const void* k_cache, const void* v_cache, int64_t num_pages,
                                       const int32_t* block_tables, int32_t max_pages_per_seq,
                                       const int32_t* seq_lens, const int32_t* cu_seqlens_q,
                                       int32_t num_seqs, int32_t total_q, int32_t num_q_heads,
                                       int32_t num_kv_heads, const float* k_descale,
                                       const float* v_descale, float softmax_scale,
                                       int32_t num_segments, void* out, int64_t out_stride_tok,
                                       int64_t out_stride_head, int32_t* status, void* stream);

/*
 * Scheduling switch for later calls: 1 = fixed page ranges per piece
 * (bit-identical results across calls), 0 = balanced tile sharing (the default;
 * see the top of this file).  Thread-safe; takes effect at the next launch.
 * The switch is PROCESS-WIDE: it changes the results' bit pattern (not their
 * accuracy) for every caller of the library in the process, on every thread and
 * device, so a library that needs bit-identical repeats should set it once at
 * start-up rather than around its own calls.  No counterpart on the pages.
 */
void mtp_verify_attn_set_deterministic(int32_t on);
int32_t mtp_verify_attn_get_deterministic(void);

/*
 * How the split-KV pieces are laid out over the SMs (process-wide switch):
 *  - MTPATTN_SCHED_PLANNED (the default; used when the batch has at most 256
 *    (sequence, KV head) units and no more units than SMs, else chunked): the
 *    main kernel first reads seq_lens and gives each unit a number of pieces in
 *    proportion to its length, so ragged batches keep every SM streaming.  With
 *    equal lengths it lays the pieces out exactly as chunked scheduling does.
 *  - MTPATTN_SCHED_CHUNKED: from the host-side shape alone, every unit is cut as
 *    if it held max_pages pages; short sequences leave their SMs idle.
 * Returns MTPATTN_E_ARG for an unknown mode.  Thread-safe; takes effect at the
 * next launch.  Like the deterministic switch it is PROCESS-WIDE: it selects the
 * kernel (and the num_segments heuristic) for every caller in the process.  No
 * counterpart on the pages, which leave the split of a sequence open.
 */
#define MTPATTN_SCHED_CHUNKED 0
#define MTPATTN_SCHED_PLANNED 1
int32_t mtp_verify_attn_set_scheduling(int32_t mode);
int32_t mtp_verify_attn_get_scheduling(void);

/* Static description of a status code (never NULL).  The library's own; no counterpart
 * on the pages. */
const char* mtp_verify_attn_strerror(int status);

/*
 * Streaming-read ceiling probe (the device's practical read bandwidth, measured
 * the way the aiter PR #5190 page quotes its 5.9-6.9 TB/s ceiling): every byte
 * of the device buffer `buf` (`bytes`, a multiple of 16, 16-byte aligned) is
 * read once with 16-byte loads by `blocks` CTAs (0 = 2 per SM) and folded into
 * one uint32 per CTA written to device `sink` [blocks], so the reads are not
 * dead code.  One kernel launch on `stream`.
 */
int mtpattn_stream_read(const void* buf, size_t bytes, uint32_t* sink, int32_t blocks,
                        void* stream);

/* Number of CTAs mtpattn_stream_read launches for blocks = 0 on the current device. */
int32_t mtpattn_stream_read_default_blocks(void);

#ifdef __cplusplus
}
#endif

#endif /* MTPATTN_H */
