"""dsa_index_score_prefill: index scores of query rows given by row ranges.  Four
consecutive rows share each key tile where they start at the same key (a
"shared" group: causal rows of one segment); a group with a segment boundary
inside it, or rows with unrelated ranges, is "split" and walks each row's own
tiles.  Every case is checked against the oracle's per-row definition of the
score (the DSA lightning indexer, the "scores" stage of tokenspeed PR #627):
bit-exact on integer-grid bf16 inputs, whose fp32 scores are exact; within a
relative 1e-5 on fp8 inputs."""
import numpy as np
import pytest
import torch

from deepseek_sparse_attention_index_gb300 import build as B
from deepseek_sparse_attention_index_gb300 import inputs as I
from deepseek_sparse_attention_index_gb300 import ops
from oracle import dsa_oracle as O
from tests.helpers import raw

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    B.build()
    ops.load()


def _ind_np(ind):
    return dict(q_idx=raw(ind["q_idx"]), q_scale=raw(ind["q_scale"]), k_idx=raw(ind["k_idx"]),
                k_scale=raw(ind["k_scale"]), w=raw(ind["w"]), is_fp8=ind["idx_dtype"] == 1)


def _ref(inp, t, r0, r1):
    fp8 = inp["is_fp8"]
    q = O.index_values(inp["q_idx"][t], inp["q_scale"][t] if fp8 else None, fp8)
    k = O.index_values(inp["k_idx"][r0:r1], inp["k_scale"][r0:r1] if fp8 else None, fp8)
    return O.index_scores_one(q, inp["w"][t].astype(np.float64), k)


def _segments(seg_lens):
    starts, ends, s0 = [], [], 0
    for L in seg_lens:
        starts += [s0] * L
        ends += list(range(s0 + 1, s0 + L + 1))
        s0 += L
    return np.array(starts, dtype=np.int32), np.array(ends, dtype=np.int32)


def _run(ind, rs, re, max_len, flag=None):
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    return ops.dsa_index_score_prefill(ind["q_idx"], ind["idx_dtype"], ind["q_scale"],
                                       ind["k_idx"], ind["k_scale"], ind["w"], dev(rs), dev(re),
                                       max_len, err_flag=flag)


def _check_rows(sc, inp, rs, re, rows, exact):
    for t in rows:
        L = int(re[t] - rs[t])
        got = sc[t, :L].astype(np.float64)
        ref = _ref(inp, t, int(rs[t]), int(re[t]))
        if exact:
            assert np.array_equal(got, ref), t
        else:
            tol = 1e-5 * np.abs(ref).max(initial=0.0) + 1e-5 * np.abs(ref)
            assert (np.abs(got - ref) <= tol).all(), t
        assert np.isnan(sc[t, L:]).all(), t   # past the row: untouched


@pytest.mark.parametrize("H_I", [8, 32, 64])
def test_grid_segments_every_row_bit_exact(H_I):
    """Shared groups, split groups at each segment boundary (1-token segments
    included) and a partial last group (T = 993), bf16 d = 64."""
    rs, re = _segments([1, 3, 130, 257, 2, 600])
    T = len(rs)
    ind = I.indexer_grid_bf16(T, T, H_I, 64, seed=11 + H_I, device="cuda")
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    sc = _run(ind, rs, re, int((re - rs).max()), flag).cpu().numpy()
    _check_rows(sc, _ind_np(ind), rs, re, range(T), exact=True)
    assert flag.item() == 0


@pytest.mark.parametrize("H_I", [16, 64])
def test_fp8_segments_every_row(H_I):
    rs, re = _segments([1, 1, 5, 129, 500, 3])
    T = len(rs)
    ind = I.indexer_fp8(T, T, H_I, 128, seed=21 + H_I, device="cuda")
    sc = _run(ind, rs, re, int((re - rs).max())).cpu().numpy()
    _check_rows(sc, _ind_np(ind), rs, re, range(T), exact=False)


def test_unrelated_ranges_and_empty_rows():
    """Rows whose ranges share nothing (decode-like), rows of length 0, rows
    with the same start in different groups; T = 37 leaves a partial group."""
    g = np.random.default_rng(5)
    S, T = 5000, 37
    lens = g.integers(0, 700, T).astype(np.int32)
    lens[[0, 9, 10, 36]] = 0
    lens[[4, 5, 6, 7]] = [1, 128, 129, 1000]     # one group of unrelated lengths...
    rs = g.integers(0, S - 1000, T).astype(np.int32)
    rs[[12, 13, 14, 15]] = 77                    # ...and one sharing a start
    re = rs + lens
    ind = I.indexer_grid_bf16(T, S, 32, 64, seed=6, device="cuda")
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    sc = _run(ind, rs, re, int(lens.max()), flag).cpu().numpy()
    _check_rows(sc, _ind_np(ind), rs, re, range(T), exact=True)
    assert flag.item() == 0


def test_bad_range_inside_a_group_is_flagged():
    S = 300
    rs = np.array([0, 0, 0, 0, 10, 10, 250, 10], dtype=np.int32)
    re = np.array([1, 2, 3, 4, 20, 30, 301, 40], dtype=np.int32)   # row 6 runs past the cache
    ind = I.indexer_grid_bf16(8, S, 8, 64, seed=7, device="cuda")
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    sc = _run(ind, rs, re, 51, flag).cpu().numpy()
    assert flag.item() & ops.DEVERR_INDEX_RANGE
    assert np.isnan(sc[6]).all()
    _check_rows(sc, _ind_np(ind), rs, re, [0, 1, 2, 3, 4, 5, 7], exact=True)


def _sampled(T, seg_lens, seed):
    rs, re = _segments(seg_lens)
    ind = I.indexer_fp8(T, T, 64, 128, seed=seed, device="cuda")
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    sc = _run(ind, rs, re, int((re - rs).max()), flag)
    ends = np.cumsum(seg_lens)
    rows = {0, 1, 2, 3, 4, 127, 128, 129, 1000, T - 4, T - 3, T - 2, T - 1}
    rows |= {int(e) for e in ends[:-1]} | {int(e) - 1 for e in ends}   # segment edges
    rows |= set(np.random.default_rng(seed).integers(0, T, 8).tolist())
    rows = sorted(r for r in rows if 0 <= r < T)
    got = sc[torch.tensor(rows, device="cuda")].cpu().numpy()
    sub = {r: i for i, r in enumerate(rows)}
    inp = _ind_np(ind)
    for t in rows:
        L = int(re[t] - rs[t])
        ref = _ref(inp, t, int(rs[t]), int(re[t]))
        tol = 1e-5 * np.abs(ref).max() + 1e-5 * np.abs(ref)
        assert (np.abs(got[sub[t], :L].astype(np.float64) - ref) <= tol).all(), t
    assert flag.item() == 0


def test_causal_prefill_16k_full_size_sampled():
    """The causal prefill at T = 16384 (one sequence, indexer fp8 64 x 128),
    in the launch configuration the benchmark times; sampled rows."""
    _sampled(16384, [16384], seed=31)


def test_packed_segments_16k_full_size_sampled():
    """Segments with lengths drawn U[1, 8192] summing to 16384, 1-token
    segments included; rows at every segment edge are among the samples."""
    seg = I.packed_segment_lengths(16384)
    _sampled(16384, seg, seed=32)
