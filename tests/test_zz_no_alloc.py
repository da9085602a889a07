"""dsa_topk_noalloc: the top-k for callers that cannot allocate device memory.

Such callers (for example a plugin whose host framework hands it only its
input and output buffers, or a latency-critical path where cudaMalloc is not
allowed) pass no workspace; the scratch lives in a static device array inside
the library.  This file is named so that pytest collects it last.  It checks,
through the C ABI, that two calls in a row give exactly the indices of the
workspace entry point dsa_topk, and that a call too large for the static
scratch is refused on the host."""
import ctypes

import numpy as np
import pytest
import torch

from deepseek_sparse_attention_index_gb300 import build as B
from deepseek_sparse_attention_index_gb300 import ops

pytestmark = pytest.mark.gpu


def _rows(seed, T, k):
    rng = np.random.default_rng(seed)
    lens = [int(x) for x in rng.integers(1, 30000, T)]
    lens[0] = k          # exactly k
    lens[1] = 3          # fewer than k
    lens[2] = 20000      # every score tied: the candidate list overflows
    ld = (max(lens) + 3) // 4 * 4
    S = np.full((T, ld), 7.0e30, dtype=np.float32)
    for t, L in enumerate(lens):
        S[t, :L] = (np.round(rng.standard_normal(L) * 30) / 8).astype(np.float32)
    S[2, :lens[2]] = 0.25
    return torch.from_numpy(S).cuda(), torch.tensor(lens, dtype=torch.int32, device="cuda"), max(lens)


def _noalloc(scores, row_len, max_len, k, base):
    T, ld = scores.shape
    idx = torch.full((T, k), -5, dtype=torch.int32, device="cuda")
    lens = torch.full((T,), -5, dtype=torch.int32, device="cuda")
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = ops.load().dsa_topk_noalloc(
        ops._ptr(scores), ld, ops._ptr(row_len), T, int(max_len), k, ops._ptr(base),
        ops._ptr(idx), ops._ptr(lens), ops._ptr(flag), ops._stream())
    assert st == 0, ops.load().dsa_status_string(st)
    torch.cuda.synchronize()
    assert flag.item() == 0
    return idx, lens


@pytest.mark.parametrize("k", [2048, 128])
def test_noalloc_matches_workspace_topk_on_two_calls(k):
    B.build()
    T = 32
    for call, seed in enumerate([101, 202]):   # two calls in a row share the scratch
        scores, row_len, max_len = _rows(seed + k, T, k)
        base = torch.arange(T, dtype=torch.int32, device="cuda") * 100000
        ref_idx, ref_lens = ops.dsa_topk(scores, row_len, k, max_len, index_base=base)
        idx, lens = _noalloc(scores, row_len, max_len, k, base)
        assert torch.equal(idx, ref_idx), "call %d" % call
        assert torch.equal(lens, ref_lens), "call %d" % call


def test_noalloc_refuses_more_rows_than_its_scratch():
    B.build()
    T = 64                                        # 64 rows at k = 2048 need > 4 MiB
    scores = torch.zeros((T, 4096), dtype=torch.float32, device="cuda")
    row_len = torch.full((T,), 4096, dtype=torch.int32, device="cuda")
    idx = torch.empty((T, 2048), dtype=torch.int32, device="cuda")
    assert ops.dsa_topk_workspace_size(T, 4096, 2048) > (4 << 20)
    st = ops.load().dsa_topk_noalloc(ops._ptr(scores), 4096, ops._ptr(row_len), T, 4096, 2048,
                                     None, ops._ptr(idx), None, None, ops._stream())
    assert st == 2
