"""The bounded waits of the main kernel and of the segment reduce, exercised without faulting
the GPU.

A test-only build of the library (-DMTPATTN_WAIT_CYCLES=200000, about 0.1 ms of SM clocks,
and -DMTPATTN_TEST_STALL, which makes CTA 0's V producer skip its first tile) is called on a
small batch: the MMA warp's wait for that tile runs out, the CTA raises its abort flag, every
role winds down (waiting, again with a limit, for its own copies in flight), the tensor memory
is freed and the call reports MTPATTN_ERR_TIMEOUT in its status word.  The test then checks
that the GPU is still usable: a second call of the test build returns the same way, and the
product library, on the same workspace, matches the oracle.  It runs in a child process so
that the test build's kernels stay out of the other tests' process.
"""
from __future__ import annotations

import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_CHILD = textwrap.dedent("""
    import sys
    import numpy as np
    import torch
    sys.path.insert(0, {root!r})
    import oracle
    from paged_fp8_speculative_gb300 import _lib, api, synth
    from tests.helpers import oracle_args

    stall = _lib.load({path!r})
    batch = synth.make_batch([3000] * 4, 4, 16, 1, seed=31, k_descale=0.5, v_descale=2.0)
    b = batch.to("cuda")
    kd = torch.tensor([b.k_descale], dtype=torch.float32, device="cuda")
    vd = torch.tensor([b.v_descale], dtype=torch.float32, device="cuda")
    S = 8
    ws = torch.zeros(api.mtp_verify_attn_workspace_size(b.total_q, 16, S), dtype=torch.uint8,
                     device="cuda")
    out = torch.zeros_like(b.q)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(2):
        status.zero_()
        rc = stall.mtp_verify_attn_fwd(
            b.q.data_ptr(), b.q.stride(0), b.q.stride(1), b.k_cache.data_ptr(),
            b.v_cache.data_ptr(), b.k_cache.shape[0], b.block_tables.data_ptr(),
            b.block_tables.shape[1], b.seq_lens.data_ptr(), b.cu_seqlens_q.data_ptr(),
            b.num_seqs, b.total_q, 16, 1, kd.data_ptr(), vd.data_ptr(), b.softmax_scale, S,
            ws.data_ptr(), ws.numel(), out.data_ptr(), out.stride(0), out.stride(1),
            status.data_ptr(), torch.cuda.current_stream().cuda_stream)
        assert rc == 0, rc
        torch.cuda.synchronize()                      # the call returned
        assert status.item() & api.ERR_TIMEOUT, status.item()
        assert ws[:4096].count_nonzero().item() == 0  # the reduce still reset the counters
    # the product library on the same workspace, with its normal wait limit
    status.zero_()
    got = api.mtp_verify_attn_fwd(b.q, b.k_cache, b.v_cache, b.block_tables, b.seq_lens,
                                  b.cu_seqlens_q, kd, vd, b.softmax_scale, num_segments=S,
                                  workspace=ws, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0, status.item()
    ref = oracle.verify_attention(*oracle_args(batch))
    err = oracle.excess_over_half_ulp(got.float().cpu().numpy().astype(np.float64), ref)
    assert err <= 0.01, err
    print("wait-limit test ok", err)
""")


@pytest.fixture(scope="module")
def stall_lib():
    """The test-only build (short wait limit, CTA 0 skipping its first V tile), built once."""
    from paged_fp8_speculative_gb300 import build
    path = os.path.join(build.BUILD, "libmtpattn_stall.so")
    build.build(extra_flags=("-DMTPATTN_WAIT_CYCLES=200000", "-DMTPATTN_TEST_STALL=1"),
                lib_path=path)
    return path


def test_pipeline_wait_limit_returns_timeout_status(stall_lib):
    r = subprocess.run([sys.executable, "-c", _CHILD.format(root=ROOT, path=stall_lib)],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr


_PREFILL_CHILD = textwrap.dedent("""
    import ctypes, sys
    import torch
    sys.path.insert(0, {root!r})
    from paged_fp8_speculative_gb300 import _lib, api, synth

    stall = _lib.load({path!r})
    lq, lk = [300, 200], [700, 260]
    b = synth.make_prefill_batch(lq, lk, 4, 2, seed=33).to("cuda")
    H = 4
    desc = [torch.tensor([x], dtype=torch.float32, device="cuda")
            for x in (b.q_descale, b.k_descale, b.v_descale)]
    ref = api.fmha_fwd_fp8_varlen(b.q, b.k, b.v, *desc, b.cu_seqlens_q, b.cu_seqlens_k,
                                  max(lq), max(lk))
    torch.cuda.synchronize()
    for _ in range(2):
        out = torch.full_like(ref, 7.0)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        rc = stall.fmha_fwd_fp8_varlen(
            b.q.data_ptr(), b.q.stride(0), b.q.stride(1), b.k.data_ptr(), b.k.stride(0),
            b.k.stride(1), b.v.data_ptr(), b.v.stride(0), b.v.stride(1),
            b.cu_seqlens_q.data_ptr(), b.cu_seqlens_k.data_ptr(), len(lq), sum(lq), sum(lk),
            max(lq), max(lk), H, 2, desc[0].data_ptr(), desc[1].data_ptr(), desc[2].data_ptr(),
            ctypes.c_float(1.0 / 192 ** 0.5), 0, out.data_ptr(), out.stride(0), out.stride(1),
            None, status.data_ptr(), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert rc == 0, rc
        torch.cuda.synchronize()                      # the call returned
        assert status.item() & api.ERR_TIMEOUT, status.item()
        # CTA 0 (the first 128 queries of sequence 0, head 0) gave up without writing;
        # every other row is the product library's
        assert bool((out[:128, 0] == 7.0).all())
        keep = torch.ones(out.shape[:2], dtype=torch.bool, device="cuda")
        keep[:128, 0] = False
        assert torch.equal(out[keep].view(torch.int16), ref[keep].view(torch.int16))
    print("prefill wait-limit test ok")
""")


def test_prefill_wait_limit_returns_timeout_status(stall_lib):
    """The prefill's bounded waits: in the test-only build, CTA 0's TMA warp never issues its
    first V tile, so the widening warps' wait for it runs out after about 0.1 ms; the CTA
    raises its abort flag, every role winds down, its tensor memory is freed and its rows are
    left unwritten, the call reports MTPATTN_ERR_TIMEOUT, and every other CTA's rows are
    exact.  A second call returns the same way (so the first freed its resources)."""
    r = subprocess.run([sys.executable, "-c", _PREFILL_CHILD.format(root=ROOT, path=stall_lib)],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "prefill wait-limit test ok" in r.stdout


def test_reduce_wait_limit_returns_timeout_status():
    """The segment reduce waits, with a limit (about 2 s of SM clocks), until the main kernel's
    CTAs have all counted themselves out of the workspace's call counters.  Two call counters
    that disagree from the start (as in a workspace whose header was not zeroed) make that
    wait run out: the call still returns, reports MTPATTN_ERR_TIMEOUT and writes zero rows,
    and once the header is zeroed again the next call on the same workspace is correct."""
    import time

    import numpy as np
    import torch

    import oracle
    from paged_fp8_speculative_gb300 import api, synth
    from tests.helpers import oracle_args

    batch = synth.make_batch([3000] * 4, 4, 16, 1, seed=32, k_descale=0.5, v_descale=2.0)
    b = batch.to("cuda")
    kd = torch.tensor([b.k_descale], dtype=torch.float32, device="cuda")
    vd = torch.tensor([b.v_descale], dtype=torch.float32, device="cuda")
    S = 8
    ws = torch.zeros(api.mtp_verify_attn_workspace_size(b.total_q, 16, S), dtype=torch.uint8,
                     device="cuda")
    ws[4100:4104].view(torch.int32).fill_(12345)          # "finished" never equals "started"
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.time()
    out = api.mtp_verify_attn_fwd(b.q, b.k_cache, b.v_cache, b.block_tables, b.seq_lens,
                                  b.cu_seqlens_q, kd, vd, b.softmax_scale, num_segments=S,
                                  workspace=ws, status=status)
    torch.cuda.synchronize()
    assert time.time() - t0 < 60
    assert status.item() & api.ERR_TIMEOUT, status.item()
    assert out.abs().max().item() == 0
    ws.zero_()
    status.zero_()
    got = api.mtp_verify_attn_fwd(b.q, b.k_cache, b.v_cache, b.block_tables, b.seq_lens,
                                  b.cu_seqlens_q, kd, vd, b.softmax_scale, num_segments=S,
                                  workspace=ws, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0, status.item()
    ref = oracle.verify_attention(*oracle_args(batch))
    assert oracle.excess_over_half_ulp(got.float().cpu().numpy().astype(np.float64), ref) <= 0.01
