// The fp8 Q/P tier of the split-KV main kernel: the planned-scheduling kernel of
// attn_main_planned.cu compiled a second time with MTPATTN_QP_FP8 set, so that Q and P are
// each rounded once to e4m3 (aiter PR #5190 page, "Kernel notes": the pages' kernel quantizes
// Q and P to fp8) instead of being carried as two e4m3 terms.  Layout, scheduling, MMAs and
// the segment reduce are those of the default kernel; only the two roundings differ (see
// attn_main_common.cuh).  The kernel and its launch function get names of their own.
#define MTPATTN_QP_FP8 1
#define attn_main_planned_kernel attn_main_planned_qp8_kernel
#define launch_attn_main_planned launch_attn_main_planned_qp8
#define MTPATTN_COVERAGE_READER mtpattn_test_coverage_planned_qp8
#include "attn_main_planned.cu"
