"""Index and page coverage of the split-KV main kernel, counted exactly.

A test-only build of the library (-DMTPATTN_TEST_COVERAGE) counts, in a device array, every
(sequence, KV head, logical page) whose K the main kernel streams, at the page whose block-
table entry it actually reads.  Whatever the scheduling (planned or chunked), the tile mode
(balanced sharing or fixed ranges), the segment count (1 to 64, or the library's choice with
its slot pool) and the batch (ragged q_len, empty-tail segments, several KV heads, more units
than SMs), each of a sequence's ceil(L / 16) pages must be streamed exactly once and no
other page at all: a missed page, a page taken twice by two pieces, or a read past a
sequence's last page shows up as a count other than 1 or 0.  The outputs are also checked
against the oracle.  It runs in a child process so that the test build's kernels stay out of
the other tests' process.
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
    import ctypes, sys
    import numpy as np
    import torch
    sys.path.insert(0, {root!r})
    import oracle
    from paged_fp8_speculative_gb300 import _lib, api, synth
    from tests.helpers import oracle_args

    cov = _lib.load({path!r})
    readers = []
    for name in ("mtpattn_test_coverage_planned", "mtpattn_test_coverage_chunked"):
        fn = getattr(cov, name)
        fn.restype = ctypes.c_int
        fn.argtypes = [ctypes.c_void_p, ctypes.c_int64]
        readers.append(fn)

    def counts(n):
        total = np.zeros(n, dtype=np.uint32)
        buf = np.zeros(n, dtype=np.uint32)
        for fn in readers:
            assert fn(buf.ctypes.data, n) == 0
            total += buf
        return total

    BATCHES = {{
        "ragged_extend": lambda: synth.make_batch([6, 17, 250, 1031, 4099, 33], [1, 4, 2, 3, 4, 1],
                                                  16, 1, seed=61, k_descale=0.5, v_descale=2.0),
        "decode_kv2": lambda: synth.make_batch([1, 2, 300, 1500, 16, 17], 1, 32, 2, seed=62),
        "one_long": lambda: synth.make_batch([20000, 40, 3], [4, 2, 1], 16, 1, seed=63, spare_pages=5),
        "tail_segments": lambda: synth.make_batch([8000] * 4, 4, 16, 1, seed=64),
        "many_units": lambda: synth.make_batch([40 + 37 * (i % 11) for i in range(180)], 1, 16, 1,
                                               seed=65),
    }}
    checked = 0
    for name, mk in BATCHES.items():
        batch = mk()
        b = batch.to("cuda")
        hkv = b.num_kv_heads
        mp = b.block_tables.shape[1]
        n = b.num_seqs * hkv * mp
        want = np.zeros((b.num_seqs, hkv, mp), dtype=np.uint32)
        for s, L in enumerate(batch.seq_lens.tolist()):
            want[s, :, :(L + 15) // 16] = 1
        ref = oracle.verify_attention(*oracle_args(batch))
        kd = torch.tensor([b.k_descale], dtype=torch.float32, device="cuda")
        vd = torch.tensor([b.v_descale], dtype=torch.float32, device="cuda")
        for sched in (api.SCHED_PLANNED, api.SCHED_CHUNKED):
            cov.mtp_verify_attn_set_scheduling(sched)
            for det in (0, 1):
                cov.mtp_verify_attn_set_deterministic(det)
                for S in (0, 1, 3, 16, 64):
                    Sr = S or cov.mtp_verify_attn_num_segments(b.num_seqs, hkv, mp, -1)
                    ws = torch.zeros(api.mtp_verify_attn_workspace_size(b.total_q, b.num_q_heads, Sr),
                                     dtype=torch.uint8, device="cuda")
                    out = torch.zeros_like(b.q)
                    status = torch.zeros(1, dtype=torch.int32, device="cuda")
                    counts(n)                          # clear
                    rc = cov.mtp_verify_attn_fwd(
                        b.q.data_ptr(), b.q.stride(0), b.q.stride(1), b.k_cache.data_ptr(),
                        b.v_cache.data_ptr(), b.k_cache.shape[0], b.block_tables.data_ptr(), mp,
                        b.seq_lens.data_ptr(), b.cu_seqlens_q.data_ptr(), b.num_seqs, b.total_q,
                        b.num_q_heads, hkv, kd.data_ptr(), vd.data_ptr(), b.softmax_scale, S,
                        ws.data_ptr(), ws.numel(), out.data_ptr(), out.stride(0), out.stride(1),
                        status.data_ptr(), torch.cuda.current_stream().cuda_stream)
                    assert rc == 0, (name, sched, det, S, rc)
                    torch.cuda.synchronize()
                    assert status.item() == 0, (name, sched, det, S, status.item())
                    got = counts(n).reshape(b.num_seqs, hkv, mp)
                    bad = np.argwhere(got != want)
                    assert bad.size == 0, (name, sched, det, S, bad[:5].tolist(),
                                           [int(got[tuple(i)]) for i in bad[:5]])
                    err = oracle.excess_over_half_ulp(out.float().cpu().numpy().astype(np.float64), ref)
                    assert err <= 0.01, (name, sched, det, S, err)
                    checked += 1
    print("coverage ok", checked)
""")


def test_every_page_streamed_exactly_once():
    from paged_fp8_speculative_gb300 import build
    path = os.path.join(build.BUILD, "libmtpattn_coverage.so")
    build.build(extra_flags=("-DMTPATTN_TEST_COVERAGE=1",), lib_path=path)
    r = subprocess.run([sys.executable, "-c", _CHILD.format(root=ROOT, path=path)], cwd=ROOT,
                       capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "coverage ok 100" in r.stdout, r.stdout
