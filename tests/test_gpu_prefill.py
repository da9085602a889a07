"""Causal prefill end to end through the C ABI, at the sizes of the prefill
workload: single sequences of T = 4096, 16384 and 65536 tokens and a packed
batch of segments with lengths U[1, 8192] summing to 16384 (1-token segments
included); indexer 64 heads x 128 fp8, top-k 2048 (-1 padding for the first
2047 tokens of a segment), sparse MLA at H = 8, 16 and 64 over bf16 rows of
576 (miles PR #3608 "per-arch DSA sparse attention dispatch", Correctness:
packed sequences end to end, causal ranges -> indexer -> top-k -> attention).

Each case runs dsa_index_score_prefill -> dsa_topk -> dsa_sparse_mla_fwd on
the GPU.  The oracle recomputes the chosen query rows one by one from the
same tensors: every row at T = 4096, sampled rows otherwise (the first
tokens, the rows around the 2048 padding edge, every segment's first, second
and last token, and seeded random rows)."""
import numpy as np
import pytest
import torch

import oracle.dsa_oracle as O
from deepseek_sparse_attention_index_gb300 import build as B
from deepseek_sparse_attention_index_gb300 import inputs as I
from deepseek_sparse_attention_index_gb300 import ops
from tests.helpers import raw, pool_np
from tests.parity import check_index_sets, check_out_lse

pytestmark = pytest.mark.gpu

HEADS = (8, 16, 64)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    B.build()
    ops.load()


def _pipeline(case):
    """index score (causal rows) -> top-k on the GPU; returns idx (global
    slots, -1 padded) and lens."""
    ind = case.indexer
    maxL = int((case.row_end - case.row_start).max())
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    sc = ops.dsa_index_score_prefill(ind["q_idx"], ind["idx_dtype"], ind["q_scale"], ind["k_idx"],
                                     ind["k_scale"], ind["w"], case.row_start, case.row_end, maxL,
                                     err_flag=flag)
    rl = (case.row_end - case.row_start).contiguous()
    idx, lens = ops.dsa_topk(sc, rl, case.k, maxL, index_base=case.row_start, err_flag=flag)
    torch.cuda.synchronize()
    del sc
    assert flag.item() == 0
    return idx, lens


class _Oracle:
    """The oracle's steps for chosen query rows, with the index keys and the KV
    pool decoded once for the whole sequence."""

    def __init__(self, case):
        ind = case.indexer
        self.fp8 = ind["idx_dtype"] == I.IDX_FP8
        self.q_idx = raw(ind["q_idx"])
        self.q_scale = raw(ind["q_scale"])
        self.w = raw(ind["w"])
        self.kvals = O.index_values(raw(ind["k_idx"]), raw(ind["k_scale"]) if self.fp8 else None,
                                    self.fp8)
        self.kv_all = O.kv_rows(pool_np(case.kv), np.arange(case.T))
        self.r0 = raw(case.row_start).astype(np.int64)
        self.r1 = raw(case.row_end).astype(np.int64)
        self.k = case.k

    def select(self, t):
        q_t = O.index_values(self.q_idx[t], self.q_scale[t] if self.fp8 else None, self.fp8)
        scores = O.index_scores_one(q_t, self.w[t].astype(np.float64),
                                    self.kvals[self.r0[t]:self.r1[t]])
        return scores, O.topk_row(scores, self.k)


def _check(case, rows, heads=HEADS):
    idx, lens = _pipeline(case)
    ref = _Oracle(case)
    rows = sorted(set(int(t) for t in rows if 0 <= t < case.T))
    sel = torch.tensor(rows, dtype=torch.long, device="cuda")
    idx_np = idx[sel].cpu().numpy()
    lens_np = lens[sel].cpu().numpy()
    # the selection: count, -1 tail, the set (bit-exact up to tolerated ties)
    attn_rows = {}
    for i, t in enumerate(rows):
        L = int(ref.r1[t] - ref.r0[t])
        n = min(L, case.k)
        assert lens_np[i] == n, t
        assert (idx_np[i, :n] >= 0).all() and (idx_np[i, n:] == -1).all(), t
        pos = np.where(idx_np[i] >= 0, idx_np[i] - ref.r0[t], -1)
        assert (pos[:n] < L).all(), t
        scores, ref_sel = ref.select(t)
        gset = check_index_sets(pos, ref_sel, scores, case.k)
        use = np.sort(ref_sel[:n]) if gset is None else gset
        attn_rows[t] = ref.kv_all[use + ref.r0[t]]
    # attention at each head count over the same selection
    for H in heads:
        q = I.prefill_q(case.T, H, device="cuda")
        flag = torch.zeros(1, dtype=torch.int32, device="cuda")
        out, lse = ops.dsa_sparse_mla_fwd(q, case.softmax_scale, case.kv, idx, err_flag=flag)
        torch.cuda.synchronize()
        assert flag.item() == 0
        q_np = raw(q[sel])
        out_np = out[sel].float().cpu().numpy()
        lse_np = lse[sel].cpu().numpy()
        del q, out, lse
        for i, t in enumerate(rows):
            ref_out, ref_lse = O.sparse_mla_one(O.decode_bf16(q_np[i]), attn_rows[t],
                                                case.softmax_scale, 512)
            check_out_lse(out_np[i], lse_np[i], ref_out, ref_lse, "H=%d token %d" % (H, t))


def _edge_rows(seg_lens):
    rows = []
    s0 = 0
    for L in seg_lens:
        for off in (0, 1, 2, 2045, 2046, 2047, 2048, 2049, L // 2, L - 2, L - 1):
            if 0 <= off < L:
                rows.append(s0 + off)
        s0 += L
    return rows


def _random_rows(T, n, seed):
    return list(np.random.default_rng(seed).integers(0, T, n))


def test_prefill_t4096_every_row():
    case = I.prefill_case([4096], H=8, device="cuda", name="prefill_T4096")
    _check(case, range(4096))


@pytest.mark.parametrize("T", [16384, 65536])
def test_prefill_long_sampled_rows(T):
    case = I.prefill_case([T], H=8, device="cuda", name="prefill_T%d" % T)
    rows = _edge_rows([T]) + [4095, 4096, 8191, 8192, 16383, T - 3] + _random_rows(T, 16, T)
    _check(case, rows)


def test_prefill_packed_16k_segments():
    lens = I.packed_segment_lengths()
    assert sum(lens) == 16384 and lens.count(1) >= 2
    case = I.prefill_case(lens, H=8, device="cuda", name="prefill_packed16k")
    _check(case, _edge_rows(lens) + _random_rows(case.T, 24, 7))
