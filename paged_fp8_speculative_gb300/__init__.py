"""Paged fp8 split-KV attention for speculative-decoding verify, draft extend and
decode on GB300 (sm_103a): a C-ABI CUDA library (libmtpattn.so) and its thin
Python binding.  The attention entry points load the library on first use and
raise if it has not been built."""
from .api import (MtpAttnError, mtp_verify_attn_fwd, mtp_verify_attn_num_segments,
                  mtp_verify_attn_strerror, mtp_verify_attn_workspace_size, mtpattn_stream_read)

__all__ = ["MtpAttnError", "mtp_verify_attn_fwd", "mtp_verify_attn_num_segments",
           "mtp_verify_attn_strerror", "mtp_verify_attn_workspace_size", "mtpattn_stream_read"]
