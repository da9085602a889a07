"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Small cases are compared element by element; the full-size workloads are
compared on sampled requests the oracle computes one by one."""
import math

import numpy as np
import pytest
import torch

import oracle.dsa_oracle as O
from deepseek_sparse_attention_index_gb300 import build as B
from deepseek_sparse_attention_index_gb300 import inputs as I
from deepseek_sparse_attention_index_gb300 import ops
from tests.helpers import raw, pool_np, decode_case_np, prefill_case_np
from tests.parity import check_index_sets, check_out_lse, lse_tol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    B.build()
    ops.load()


def _flag():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


# ---------------------------------------------------------------- index score

def _oracle_scores(ind_np, t, r0, r1):
    fp8 = ind_np["is_fp8"]
    q = O.index_values(ind_np["q_idx"][t], None if not fp8 else ind_np["q_scale"][t], fp8)
    k = O.index_values(ind_np["k_idx"][r0:r1], None if not fp8 else ind_np["k_scale"][r0:r1], fp8)
    return O.index_scores_one(q, ind_np["w"][t].astype(np.float64), k)


def _ind_np(ind):
    return dict(q_idx=raw(ind["q_idx"]), q_scale=raw(ind["q_scale"]), k_idx=raw(ind["k_idx"]),
                k_scale=raw(ind["k_scale"]), w=raw(ind["w"]), is_fp8=ind["idx_dtype"] == 1)


@pytest.mark.parametrize("H_I,d", [(8, 64), (16, 128), (64, 128)])
def test_index_score_integer_grid_bit_exact(H_I, d):
    lens = [1, 127, 128, 129, 3000]
    S = sum(lens)
    ind = I.indexer_grid_bf16(len(lens), S, H_I, d, seed=1, device="cuda")
    starts = np.cumsum([0] + lens[:-1])
    rs = torch.tensor(starts, dtype=torch.int32, device="cuda")
    re = torch.tensor(starts + np.array(lens), dtype=torch.int32, device="cuda")
    flag = _flag()
    sc = ops.dsa_index_score(ind["q_idx"], 0, None, ind["k_idx"], None, ind["w"], rs, re, max(lens),
                             err_flag=flag)
    sc = sc.cpu().numpy()
    inp = _ind_np(ind)
    for t, L in enumerate(lens):
        ref = _oracle_scores(inp, t, starts[t], starts[t] + L)
        assert np.array_equal(sc[t, :L].astype(np.float64), ref), t
        assert np.isnan(sc[t, L:]).all()    # past the row: untouched
    assert flag.item() == 0


def test_index_score_causal_rows_bit_exact():
    """One causal segment (row t sees keys [0, t]): consecutive rows are scored
    against shared key tiles, each keeping its own range; odd T leaves a
    partial last group."""
    T = 1001
    ind = I.indexer_grid_bf16(T, T, 64, 128, seed=3, device="cuda")
    rs = torch.zeros(T, dtype=torch.int32, device="cuda")
    re = torch.arange(1, T + 1, dtype=torch.int32, device="cuda")
    flag = _flag()
    sc = ops.dsa_index_score(ind["q_idx"], 0, None, ind["k_idx"], None, ind["w"], rs, re, T,
                             err_flag=flag).cpu().numpy()
    inp = _ind_np(ind)
    for t in list(range(0, T, 37)) + [126, 127, 128, 129, 255, 256, T - 2, T - 1]:
        ref = _oracle_scores(inp, t, 0, t + 1)
        assert np.array_equal(sc[t, :t + 1].astype(np.float64), ref), t
        assert np.isnan(sc[t, t + 1:]).all(), t
    assert flag.item() == 0


def test_index_score_fp8_prefill_ranges():
    case = I.prefill_case([1, 1, 100, 198, 700], k=64, H=8, device="cuda")
    ind = case.indexer
    sc = ops.dsa_index_score(ind["q_idx"], 1, ind["q_scale"], ind["k_idx"], ind["k_scale"],
                             ind["w"], case.row_start, case.row_end, 700).cpu().numpy()
    inp = _ind_np(ind)
    rs, re = raw(case.row_start), raw(case.row_end)
    for t in list(range(0, case.T, 7)) + [case.T - 1]:
        ref = _oracle_scores(inp, t, rs[t], re[t])
        got = sc[t, :re[t] - rs[t]].astype(np.float64)
        tol = 1e-5 * np.abs(ref).max() + 1e-5 * np.abs(ref)
        assert (np.abs(got - ref) <= tol).all(), t


def test_index_score_flags_bad_ranges():
    ind = I.indexer_grid_bf16(2, 100, 8, 64, seed=2, device="cuda")
    rs = torch.tensor([0, 50], dtype=torch.int32, device="cuda")
    re = torch.tensor([10, 101], dtype=torch.int32, device="cuda")   # row 1 runs past k_rows
    flag = _flag()
    sc = ops.dsa_index_score(ind["q_idx"], 0, None, ind["k_idx"], None, ind["w"], rs, re, 51,
                             err_flag=flag).cpu().numpy()
    assert flag.item() & ops.DEVERR_INDEX_RANGE
    assert np.isnan(sc[1]).all() and not np.isnan(sc[0, :10]).any()


# ---------------------------------------------------------------- top-k

def _run_topk(rows, k, base=None):
    T = len(rows)
    maxL = max(max(len(r) for r in rows), 1)
    ld = (maxL + 3) // 4 * 4
    S = np.zeros((T, ld), dtype=np.float32)
    for t, r in enumerate(rows):
        S[t, :len(r)] = r
        S[t, len(r):] = np.float32(1e30)     # beyond the row: must be ignored
    sc = torch.from_numpy(S).cuda()
    rl = torch.tensor([len(r) for r in rows], dtype=torch.int32, device="cuda")
    bt = None if base is None else torch.tensor(base, dtype=torch.int32, device="cuda")
    flag = _flag()
    idx, lens = ops.dsa_topk(sc, rl, k, maxL, index_base=bt, err_flag=flag)
    assert flag.item() == 0
    return idx.cpu().numpy(), lens.cpu().numpy()


@pytest.mark.parametrize("k", [1, 7, 128, 2048])
def test_topk_bit_exact(k):
    rng = np.random.default_rng(k)
    rows = [np.zeros(0, np.float32),
            rng.standard_normal(1).astype(np.float32),
            (np.round(rng.standard_normal(k) * 8) / 4).astype(np.float32),
            (np.round(rng.standard_normal(k + 1) * 8) / 4).astype(np.float32),
            rng.standard_normal(3 * k + 5).astype(np.float32),
            (np.round(rng.standard_normal(70001) * 40) / 8).astype(np.float32),
            np.full(20000, 0.5, np.float32),                      # every score tied
            np.where(rng.random(5000) < 0.5, -0.0, 0.0).astype(np.float32),
            (-np.abs(rng.standard_normal(9000)) * 1e-30).astype(np.float32)]
    base = [int(x) for x in rng.integers(0, 1000, len(rows))]
    idx, lens = _run_topk(rows, k, base)
    for t, r in enumerate(rows):
        ref = O.topk_row(r.astype(np.float64), k)
        n = min(len(r), k)
        assert lens[t] == n
        got = idx[t]
        assert (got[n:] == -1).all()
        assert np.array_equal(got[:n], np.sort(ref[:n]) + base[t]), t   # ascending positions


def test_topk_random_fp32_many_rows():
    rng = np.random.default_rng(11)
    rows = [rng.standard_normal(int(L)).astype(np.float32) * rng.uniform(0.01, 100)
            for L in rng.integers(1, 40000, 48)]
    idx, lens = _run_topk(rows, 2048)
    for t, r in enumerate(rows):
        ref = O.topk_row(r.astype(np.float64), 2048)
        n = min(len(r), 2048)
        assert np.array_equal(idx[t, :n], np.sort(ref[:n]))


def test_topk_more_rows_than_a_grid_dimension():
    # 65537 rows (prefill at 64K tokens has as many): rows and chunks share
    # one grid dimension, so the row count is not capped at 65535
    rng = np.random.default_rng(7)
    T, k = 65537, 8
    lens = rng.integers(0, 40, T)
    rows = [(np.round(rng.standard_normal(int(L)) * 4) / 4).astype(np.float32) for L in lens]
    idx, out_lens = _run_topk(rows, k)
    for t in list(range(0, T, 997)) + [T - 1]:
        ref = O.topk_row(rows[t].astype(np.float64), k)
        n = min(len(rows[t]), k)
        assert out_lens[t] == n
        assert (idx[t, n:] == -1).all()
        assert np.array_equal(idx[t, :n], np.sort(ref[:n])), t


@pytest.mark.parametrize("k", [100, 2048])
def test_topk_long_rows_many_chunks(k):
    # rows of 8.4M-9M scores: more than 512 collect chunks each, so the ordered
    # compaction walks the chunk table in several groups; scores on a 1/64 grid
    # tie at the threshold, so the position radix runs too
    rng = np.random.default_rng(100 + k)
    rows = [(np.round(rng.standard_normal(L) * 64) / 64).astype(np.float32)
            for L in (9_000_001, 8_400_000)]
    idx, lens = _run_topk(rows, k)
    for t, r in enumerate(rows):
        ref = O.topk_row(r.astype(np.float64), k)
        assert lens[t] == k
        assert np.array_equal(idx[t], np.sort(ref[:k])), t


# ---------------------------------------------------------------- sparse MLA

def _mla_case(fmt, T, H, k, neg=0.1, seed=0, rows=4096, all_neg_row=True):
    g = torch.Generator().manual_seed(seed)
    if fmt == I.KV_BF16:
        pool = I.kv_bf16_pool(rows, seed, 5, "cuda")
        D = 576
    elif fmt == I.KV_FP8_UNIFORM:
        pool = I.kv_uniform_fp8_pool(rows, seed, 5, "cuda")
        D = 512
    else:
        pool = I.kv_packed_pool(rows, 256, seed, 5, "cuda")
        D = 512
    idx = torch.stack([torch.randperm(pool.rows, generator=g)[:k] for _ in range(T)]).to(torch.int32)
    idx[torch.rand(T, k, generator=g) < neg] = -1
    if all_neg_row and T > 1:
        idx[1] = -1
    q = I.to_bf16(torch.randn(T, H, D, generator=g)).cuda()
    return pool, idx.cuda(), q, D


@pytest.mark.parametrize("fmt,H,k", [(I.KV_BF16, 8, 300), (I.KV_BF16, 64, 2048),
                                     (I.KV_BF16, 128, 100), (I.KV_BF16, 16, 1),
                                     (I.KV_FP8_UNIFORM, 64, 1152), (I.KV_FP8_UNIFORM, 16, 77),
                                     (I.KV_FP8_DS_MLA, 64, 1024), (I.KV_FP8_DS_MLA, 8, 200)])
def test_sparse_mla_matches_oracle(fmt, H, k):
    T = 3
    pool, idx, q, D = _mla_case(fmt, T, H, k)
    scale = 1 / math.sqrt(192.0) if D == 576 else 1 / math.sqrt(512.0)
    flag = _flag()
    out, lse = ops.dsa_sparse_mla_fwd(q, scale, pool, idx, err_flag=flag)
    torch.cuda.synchronize()
    assert flag.item() == 0
    ref_out, ref_lse = O.sparse_mla(O.decode_bf16(raw(q)), pool_np(pool), raw(idx), scale,
                                    out.shape[2])
    check_out_lse(out.float().cpu().numpy(), lse.cpu().numpy(), ref_out, ref_lse, "mla",
                  lse_tol=lse_tol(fmt))
    assert (out[1] == 0).all() and torch.isneginf(lse[1]).all()   # all-padded token


def _sinks(H, seed=5):
    g = torch.Generator().manual_seed(seed)
    s = torch.randn(H, generator=g) * 3.0
    s[0] = -math.inf     # head 0: no sink
    if H > 1:
        s[1] = 40.0      # far above every score: that head's output nearly vanishes
    return s.float().cuda()


@pytest.mark.parametrize("fmt,H,k,T", [(I.KV_BF16, 64, 2048, 3),      # split pieces + combine
                                       (I.KV_BF16, 64, 256, 160),     # one piece a token
                                       (I.KV_BF16, 8, 300, 3),
                                       (I.KV_FP8_UNIFORM, 64, 1152, 3),
                                       (I.KV_FP8_DS_MLA, 64, 1024, 3)])
def test_sparse_mla_sinks(fmt, H, k, T):
    pool, idx, q, D = _mla_case(fmt, T, H, k)
    scale = 1 / math.sqrt(192.0) if D == 576 else 1 / math.sqrt(512.0)
    sinks = _sinks(H)
    out, lse = ops.dsa_sparse_mla_fwd(q, scale, pool, idx, sinks=sinks)
    ref_out, ref_lse = O.sparse_mla(O.decode_bf16(raw(q)), pool_np(pool), raw(idx), scale,
                                    out.shape[2], sinks=sinks.double().cpu().numpy())
    check_out_lse(out.float().cpu().numpy(), lse.cpu().numpy(), ref_out, ref_lse, "mla+sinks",
                  lse_tol=lse_tol(fmt))
    # the all-padded token: no value, the denominator is the sink alone
    assert (out[1] == 0).all()
    assert torch.equal(lse[1].cpu(), sinks.cpu())



def _vmax(pool, idx, Dv):
    """[T, 1, Dv]: the largest |V[d]| over each token's valid selected rows."""
    pnp, ix = pool_np(pool), raw(idx)
    vm = np.zeros((ix.shape[0], 1, Dv))
    for t in range(ix.shape[0]):
        sl = ix[t][ix[t] >= 0].astype(np.int64)
        if sl.size:
            vm[t, 0] = np.abs(O.kv_rows(pnp, sl)[:, :Dv]).max(axis=0)
    return vm


@pytest.mark.parametrize("fmt,T,H,k", [(I.KV_BF16, 32, 64, 2048),      # 4 pieces a token
                                       (I.KV_BF16, 40, 64, 600),       # 3 pieces
                                       (I.KV_BF16, 64, 32, 300),       # 2 pieces, 32 heads
                                       (I.KV_FP8_UNIFORM, 32, 64, 1152),
                                       (I.KV_FP8_DS_MLA, 40, 16, 700)])
def test_sparse_mla_few_pieces_a_token(fmt, T, H, k):
    # Batches of 32-76 tokens split each list into 2-4 pieces (one wave of
    # CTAs), whose partials the combine merges: with sinks and log2 lse, and
    # a token whose list is all -1 (its pieces are empty: no value, lse = the
    # sink).  The packed pool is held to its logit-error bound
    # (tests/parity.py): at these batch sizes some of its small output
    # elements exceed the unit-scale one.
    pool, idx, q, D = _mla_case(fmt, T, H, k)
    scale = 1 / math.sqrt(192.0) if D == 576 else 1 / math.sqrt(512.0)
    Dv = 512 if D == 576 else 448
    # the pieces a token, read off the partials' workspace (T x pieces x H records)
    pieces = round(ops.dsa_sparse_mla_workspace_size(T, H, Dv, k) / (T * H * (Dv + 1) * 4))
    assert 2 <= pieces <= 4, pieces
    ref_out, ref_lse = O.sparse_mla(O.decode_bf16(raw(q)), pool_np(pool), raw(idx), scale, Dv)
    vmax = _vmax(pool, idx, Dv) if fmt == I.KV_FP8_DS_MLA else None
    flag = _flag()
    out, lse = ops.dsa_sparse_mla_fwd(q, scale, pool, idx, err_flag=flag)
    torch.cuda.synchronize()
    assert flag.item() == 0
    check_out_lse(out.float().cpu().numpy(), lse.cpu().numpy(), ref_out, ref_lse, "pieces",
                  lse_tol=lse_tol(fmt), vmax=vmax)
    sinks = _sinks(H)
    out, lse = ops.dsa_sparse_mla_fwd(q, scale, pool, idx, sinks=sinks, lse_log2=True)
    ref_out, ref_lse = O.sparse_mla(O.decode_bf16(raw(q)), pool_np(pool), raw(idx), scale,
                                    out.shape[2], sinks=sinks.double().cpu().numpy())
    check_out_lse(out.float().cpu().numpy(), lse.cpu().numpy() * math.log(2.0), ref_out, ref_lse,
                  "pieces+sinks", lse_tol=lse_tol(fmt), vmax=vmax)
    assert (out[1] == 0).all()
    assert torch.allclose(lse[1].cpu() * math.log(2.0), sinks.cpu(), rtol=1e-6, atol=1e-6)

def test_sparse_mla_lse_log2():
    pool, idx, q, D = _mla_case(I.KV_BF16, 3, 64, 700)
    scale = 1 / math.sqrt(192.0)
    out, lse = ops.dsa_sparse_mla_fwd(q, scale, pool, idx)
    out2, lse2 = ops.dsa_sparse_mla_fwd(q, scale, pool, idx, lse_log2=True)
    assert torch.equal(out, out2)
    fin = torch.isfinite(lse)
    assert torch.equal(torch.isneginf(lse2), torch.isneginf(lse))
    assert torch.allclose(lse2[fin], lse[fin] / math.log(2.0), rtol=1e-6, atol=1e-6)


def test_decode_sinks_and_log2_lse():
    case = I.decode_case("sinks", 3, [300, 5000, 20000], 64, 128, "fp8", 2048, 64, I.KV_BF16,
                         device="cuda")
    sinks = _sinks(case.H)
    ind = case.indexer
    idx, out, lse = ops.dsa_decode(ind["q_idx"], ind["idx_dtype"], ind["q_scale"], ind["k_idx"],
                                   ind["k_scale"], ind["w"], case.seq_lens, case.slot_base,
                                   case.max_seq_len, case.k, case.q, case.softmax_scale, case.kv,
                                   sinks=sinks, lse_log2=True)
    idx_plain, _, _ = ops.decode_case(case)
    assert torch.equal(idx, idx_plain)          # the sinks change the attention only
    c = decode_case_np(case)
    sk = sinks.double().cpu().numpy()
    for b in range(case.B):
        rows = O.gather_valid(c["kv"], idx[b].cpu().numpy())
        ref_out, ref_lse = O.sparse_mla_one(O.decode_bf16(c["q"][b]), rows, c["softmax_scale"],
                                            c["Dv"], sk)
        check_out_lse(out[b].float().cpu().numpy(), lse[b].cpu().numpy() * math.log(2.0),
                      ref_out, ref_lse, "decode+sinks %d" % b)


def _rel_l2(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.linalg.norm(b)
    return np.linalg.norm(a - b) / den if den > 0 else np.linalg.norm(a)


@pytest.mark.parametrize("H,k,T,with_sinks", [(64, 300, 3, False), (8, 128, 4, True),
                                              (64, 2048, 2, True), (16, 100, 3, False)])
def test_sparse_mla_backward_matches_oracle(H, k, T, with_sinks):
    """Gradients of the attention (dq, the pool's row gradients, the sinks')
    against the oracle's; a small pool makes tokens share rows, token 1 is
    all -1.  Tolerance 1e-3 rel-L2: fp32 sums of up to 2048 terms on
    probabilities from the forward's lse (within 1e-4)."""
    pool, idx, q, D = _mla_case(I.KV_BF16, T, H, k, rows=2560)
    scale = 1 / math.sqrt(192.0)
    sinks = _sinks(H) if with_sinks else None
    out, lse = ops.dsa_sparse_mla_fwd(q, scale, pool, idx, sinks=sinks)
    g = torch.Generator().manual_seed(4)
    dout = I.to_bf16(torch.randn(T, H, 512, generator=g)).cuda()
    flag = _flag()
    dq, dkv, dsk = ops.dsa_sparse_mla_bwd(q, scale, pool, idx, lse, dout, sinks=sinks,
                                          err_flag=flag)
    torch.cuda.synchronize()
    assert flag.item() == 0
    sk = None if sinks is None else sinks.double().cpu().numpy()
    ref_dq, ref_dkv, ref_dsk = O.sparse_mla_bwd(O.decode_bf16(raw(q)), pool_np(pool), raw(idx),
                                                O.decode_bf16(raw(dout)), scale, 512, sk)
    assert _rel_l2(dq.cpu().numpy(), ref_dq) < 1e-3
    assert _rel_l2(dkv.cpu().numpy(), ref_dkv) < 1e-3
    assert not dq[1].any()                        # the all-padded token
    if with_sinks:
        assert _rel_l2(dsk.cpu().numpy(), ref_dsk) < 1e-3


def test_sparse_mla_backward_log2_lse_round_trip():
    pool, idx, q, D = _mla_case(I.KV_BF16, 3, 64, 400)
    scale = 1 / math.sqrt(192.0)
    dout = I.to_bf16(torch.randn(3, 64, 512, generator=torch.Generator().manual_seed(6))).cuda()
    _, lse = ops.dsa_sparse_mla_fwd(q, scale, pool, idx)
    _, lse2 = ops.dsa_sparse_mla_fwd(q, scale, pool, idx, lse_log2=True)
    a = ops.dsa_sparse_mla_bwd(q, scale, pool, idx, lse, dout)
    b = ops.dsa_sparse_mla_bwd(q, scale, pool, idx, lse2, dout, lse_log2=True)
    assert _rel_l2(b[0].cpu().numpy(), a[0].cpu().numpy()) < 1e-5
    assert _rel_l2(b[1].cpu().numpy(), a[1].cpu().numpy()) < 1e-5


def test_sparse_mla_two_loop_packed():
    T, H = 2, 64
    main = I.kv_packed_pool(T * 256, 256, 3, 6, "cuda")
    extra = I.kv_packed_pool(8192, 256, 4, 5, "cuda")
    g = torch.Generator().manual_seed(9)
    idx_main = (torch.arange(T)[:, None] * 256 + torch.arange(128)[None, :]).to(torch.int32).cuda()
    idx_extra = torch.stack([torch.randperm(8192, generator=g)[:1024] for _ in range(T)]).to(torch.int32)
    idx_extra[:, ::9] = -1
    idx_extra = idx_extra.cuda()
    q = I.to_bf16(torch.randn(T, H, 512, generator=g)).cuda()
    scale = 1 / math.sqrt(512.0)
    out, lse = ops.dsa_sparse_mla_fwd(q, scale, main, idx_main, extra, idx_extra)
    ref_out, ref_lse = O.sparse_mla(O.decode_bf16(raw(q)), pool_np(main), raw(idx_main), scale, 448,
                                    pool_np(extra), raw(idx_extra))
    check_out_lse(out.float().cpu().numpy(), lse.cpu().numpy(), ref_out, ref_lse, "2-loop",
                  lse_tol=lse_tol(I.KV_FP8_DS_MLA))


@pytest.mark.parametrize("main_fmt,extra_fmt", [(I.KV_FP8_UNIFORM, I.KV_FP8_DS_MLA),
                                               (I.KV_FP8_DS_MLA, I.KV_FP8_UNIFORM)])
def test_sparse_mla_two_loop_mixed_formats(main_fmt, extra_fmt):
    """Main and extra lists in pools of different fp8 formats (one softmax
    over both): the SIMT kernel serves these calls (the only ones the
    tensor-core kernel does not take: q must be 16-byte aligned anyway)."""
    T, H = 3, 64
    g = torch.Generator().manual_seed(21)

    def pool(fmt, rows, n):
        if fmt == I.KV_FP8_UNIFORM:
            return I.kv_uniform_fp8_pool(rows, 2, n, "cuda")
        return I.kv_packed_pool(rows, 256, 2, n, "cuda")

    main, extra = pool(main_fmt, 512, 5), pool(extra_fmt, 4096, 6)
    idx_main = torch.stack([torch.randperm(512, generator=g)[:128] for _ in range(T)]).to(torch.int32)
    idx_extra = torch.stack([torch.randperm(4096, generator=g)[:1024] for _ in range(T)]).to(torch.int32)
    idx_extra[:, ::7] = -1
    idx_main[1] = -1
    q = I.to_bf16(torch.randn(T, H, 512, generator=g)).cuda()
    scale = 1 / math.sqrt(512.0)
    flag = _flag()
    out, lse = ops.dsa_sparse_mla_fwd(q, scale, main, idx_main.cuda(), extra, idx_extra.cuda(),
                                      err_flag=flag)
    torch.cuda.synchronize()
    assert flag.item() == 0
    ref_out, ref_lse = O.sparse_mla(O.decode_bf16(raw(q)), pool_np(main), raw(idx_main), scale, 448,
                                    pool_np(extra), raw(idx_extra))
    check_out_lse(out.float().cpu().numpy(), lse.cpu().numpy(), ref_out, ref_lse, "mixed 2-loop",
                  lse_tol=lse_tol(main_fmt, extra_fmt))


def test_sparse_mla_masks_and_flags_out_of_range_entries():
    pool, idx, q, D = _mla_case(I.KV_BF16, 2, 16, 64, neg=0.0, all_neg_row=False)
    bad = idx.clone()
    bad[0, 3] = pool.rows          # one past the end
    bad[1, 5] = -7                 # below -1
    flag = _flag()
    out, lse = ops.dsa_sparse_mla_fwd(q, 0.05, pool, bad, err_flag=flag)
    assert flag.item() & ops.DEVERR_INDEX_RANGE
    masked = raw(bad).copy()
    masked[masked >= pool.rows] = -1
    masked[masked < -1] = -1
    ref_out, ref_lse = O.sparse_mla(O.decode_bf16(raw(q)), pool_np(pool), masked, 0.05, 512)
    check_out_lse(out.float().cpu().numpy(), lse.cpu().numpy(), ref_out, ref_lse, "masked")



def test_sparse_mla_uniform_extreme_scales_and_fp16_range():
    # Group scales far outside the workload's 2^[-4, 4] (2^-17, 2^-10,
    # 2^-6.9, 143, 200: products from fp16 subnormals to near its largest
    # values) still agree with the oracle; a scale that carries x s past
    # fp16's range is reported.
    pool, idx, q, D = _mla_case(I.KV_FP8_UNIFORM, 3, 64, 300, all_neg_row=False)
    sel = torch.unique(idx[idx >= 0])
    sc = pool.scales
    sc[sel[0::3], 2] = 2.0 ** -17
    sc[sel[1::5], 5] = 200.0
    sc[sel[2::7], 0] = 2.0 ** -10
    sc[sel[3::7], 3] = 2.0 ** -6.9
    sc[sel[4::9], 6] = 143.0
    scale = 1 / math.sqrt(512.0)
    flag = _flag()
    out, lse = ops.dsa_sparse_mla_fwd(q, scale, pool, idx, err_flag=flag)
    torch.cuda.synchronize()
    assert flag.item() == 0
    ref_out, ref_lse = O.sparse_mla(O.decode_bf16(raw(q)), pool_np(pool), raw(idx), scale,
                                    out.shape[2])
    check_out_lse(out.float().cpu().numpy(), lse.cpu().numpy(), ref_out, ref_lse, "scales")
    sc[sel[4], 1] = 2.0 ** 17     # any |x| > 0.5 in that group leaves fp16's range
    flag = _flag()
    ops.dsa_sparse_mla_fwd(q, scale, pool, idx, err_flag=flag)
    torch.cuda.synchronize()
    assert flag.item() & ops.DEVERR_FP16_RANGE


# ---------------------------------------------------------------- fused decode

def _check_decode(case, idx_gpu, out_gpu, lse_gpu, requests, bit_exact=False):
    c = decode_case_np(case)
    idx_gpu = idx_gpu.cpu().numpy()
    out_gpu = out_gpu.float().cpu().numpy()
    lse_gpu = lse_gpu.cpu().numpy()
    for b in requests:
        r = O.decode_request(b, c)
        if c.get("block_table") is not None:
            # paged: slot -> position through the request's pages
            page = int(c["page_size"])
            where = {int(pg): j for j, pg in enumerate(c["block_table"][b])}
            pos = np.array([where[int(s) // page] * page + int(s) % page if s >= 0 else -1
                            for s in idx_gpu[b]], dtype=np.int64)
            slots_of = lambda ps, b=b: np.array(
                [int(c["block_table"][b][p // page]) * page + p % page for p in ps], dtype=np.int64)
            base = 0
        else:
            base = int(c["slot_base"][b])
            pos = np.where(idx_gpu[b] >= 0, idx_gpu[b] - base, -1)
            slots_of = lambda ps, base=base: np.asarray(ps, dtype=np.int64) + base
        n = min(int(c["seq_lens"][b]), case.k)
        assert (pos[:n] >= 0).all() and (pos[n:] == -1).all(), b
        if bit_exact:
            assert np.array_equal(np.sort(pos[:n]), np.sort(r["idx"][:n])), b
            ref_out, ref_lse = r["out"], r["lse"]
        else:
            gset = check_index_sets(pos, r["idx"], r["scores"], case.k)
            if gset is None:
                ref_out, ref_lse = r["out"], r["lse"]
            else:   # tolerated ties: compare attention on the GPU's own selection
                rows = O.gather_valid(c["kv"], slots_of(gset))
                if c.get("idx_swa") is not None:
                    rows = np.concatenate([O.gather_valid(c["kv_swa"], c["idx_swa"][b]), rows])
                ref_out, ref_lse = O.sparse_mla_one(O.decode_bf16(c["q"][b]), rows,
                                                    c["softmax_scale"], c["Dv"])
        fmts = [case.kv.format] + ([] if case.kv_swa is None else [case.kv_swa.format])
        check_out_lse(out_gpu[b], lse_gpu[b], ref_out, ref_lse, "request %d" % b,
                      lse_tol=lse_tol(*fmts))


def test_decode_tiny_bit_exact_indices():
    case = I.tiny_decode(device="cuda")
    flag = _flag()
    idx, out, lse = ops.decode_case(case, err_flag=flag)
    torch.cuda.synchronize()
    assert flag.item() == 0
    _check_decode(case, idx, out, lse, [0], bit_exact=True)


def test_decode_ragged_fp8():
    case = I.decode_case("ragged", 5, [1, 300, 2048, 2049, 10000], 64, 128, "fp8", 2048, 64,
                         I.KV_BF16, device="cuda")
    idx, out, lse = ops.decode_case(case)
    _check_decode(case, idx, out, lse, range(5))


def test_decode_grid_ragged_many_ties_bit_exact():
    case = I.decode_case("grid", 4, [129, 700, 5000, 33000], 16, 128, "bf16_grid", 128, 16,
                         I.KV_BF16, device="cuda")
    idx, out, lse = ops.decode_case(case)
    _check_decode(case, idx, out, lse, range(4), bit_exact=True)


def test_decode_is_deterministic():
    case = I.decode_case("det", 3, [5000, 20000, 70000], 64, 128, "fp8", 2048, 64, I.KV_BF16,
                         device="cuda")
    first = [x.clone() for x in ops.decode_case(case)]
    for _ in range(5):
        again = ops.decode_case(case)
        for a, b in zip(first, again):
            assert torch.equal(a, b)


@pytest.mark.parametrize("kind,page", [("fp8", 64), ("bf16_grid", 64), ("fp8", 128)])
def test_paged_decode_matches_oracle(kind, page):
    case = I.paged_decode(4, [700, 3000, 9000, 20000], page=page, device="cuda", idx_kind=kind)
    flag = _flag()
    idx, out, lse = ops.decode_case(case, err_flag=flag)
    torch.cuda.synchronize()
    assert flag.item() == 0
    _check_decode(case, idx, out, lse, range(case.B), bit_exact=kind == "bf16_grid")


def test_paged_decode_equals_contiguous_layout():
    """The same data paged (pages shuffled, or in order) and contiguous: the
    same positions selected, the same outputs bit for bit."""
    lens = [1000, 5000, 64, 20000]
    plain = I.paged_decode(4, lens, device="cuda", shuffle=False)
    shuf = I.paged_decode(4, lens, device="cuda", shuffle=True)
    # the in-order layout through the contiguous entry point
    pages = [(L + 63) // 64 for L in lens]
    flat = I.DecodeCase(plain.name, plain.B, plain.seq_lens,
                        torch.tensor(np.cumsum([0] + [64 * n for n in pages[:-1]]),
                                     dtype=torch.int32, device="cuda"),
                        plain.max_seq_len, plain.H_I, plain.d_idx, plain.indexer, plain.k, plain.H,
                        plain.D, plain.Dv, plain.softmax_scale, plain.q, plain.kv)
    i0, o0, l0 = ops.decode_case(flat)
    i1, o1, l1 = ops.decode_case(plain)
    i2, o2, l2 = ops.decode_case(shuf)
    assert torch.equal(i0, i1) and torch.equal(o0, o1) and torch.equal(l0, l1)
    assert torch.equal(o0, o2) and torch.equal(l0, l2)
    # shuffled slots map back to the same positions
    inv = shuf.meta["new_to_old_page"]
    old = torch.where(i2 >= 0, inv.cuda()[(i2 // 64).clamp(min=0).long()] * 64 + i2 % 64, -1)
    assert torch.equal(old.to(torch.int32), i0)


def test_multi_token_decode_rows_share_a_request():
    """Q new tokens per request (speculative verification): B*Q rows that share
    their request's slot base; token i sees the context up to itself."""
    case = I.multi_token_decode(3, 4, 5000, device="cuda")
    flag = _flag()
    idx, out, lse = ops.decode_case(case, err_flag=flag)
    torch.cuda.synchronize()
    assert flag.item() == 0
    _check_decode(case, idx, out, lse, range(case.B))
    # each token's selection stays inside its own causal prefix
    pos = idx.cpu().numpy() - case.slot_base.cpu().numpy()[:, None]
    lens = case.seq_lens.cpu().numpy()
    for r in range(case.B):
        sel = pos[r][idx[r].cpu().numpy() >= 0]
        assert sel.max() < lens[r], r


def test_multi_token_decode_grid_bit_exact():
    case = I.multi_token_decode(2, 3, 3000, device="cuda", idx_kind="bf16_grid")
    idx, out, lse = ops.decode_case(case)
    _check_decode(case, idx, out, lse, range(case.B), bit_exact=True)


def _pairs_equal_single_rows(case, check_rows=(), bit_exact=False):
    """The paired index score (rows_per_request = 2) against the one-row path:
    the same selection, output and lse bit for bit; then the oracle."""
    flag = _flag()
    idx1, out1, lse1 = ops.decode_case(case, err_flag=flag)
    idx2, out2, lse2 = ops.decode_case(case, err_flag=flag, rows_per_request=2)
    torch.cuda.synchronize()
    assert flag.item() == 0
    assert torch.equal(idx1, idx2)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse1.view(torch.int32), lse2.view(torch.int32))
    if check_rows:
        _check_decode(case, idx2, out2, lse2, check_rows, bit_exact=bit_exact)


def test_multi_token_decode_pairs_equal_single_rows():
    case = I.multi_token_decode(5, 2, 20000, device="cuda", seed=3)
    _pairs_equal_single_rows(case, range(case.B))


def test_multi_token_decode_pairs_grid_bit_exact():
    # bf16 indexer of 64-wide heads (the pair path's other layout), integer grid
    case = I.multi_token_decode(3, 2, 5000, device="cuda", idx_kind="bf16_grid", d_idx=64)
    _pairs_equal_single_rows(case, range(case.B), bit_exact=True)


def test_multi_token_decode_pairs_full_size():
    """32 requests x 2 new tokens at 131072 positions (the mtp bench workload)."""
    case = I.multi_token_decode(32, 2, 131072, device="cuda")
    _pairs_equal_single_rows(case, [0, 1, 63])


def test_decode_sweep_full_size_sampled():
    """Batch 32 x 128k context, the bench workload; three requests checked."""
    case = I.decode_sweep(32, 131072, device="cuda")
    flag = _flag()
    idx, out, lse = ops.decode_case(case, err_flag=flag)
    torch.cuda.synchronize()
    assert flag.item() == 0
    _check_decode(case, idx, out, lse, [0, 17, 31])


@pytest.mark.parametrize("B,N", [(1, 512), (1, 2048), (1, 8192), (1, 32768), (1, 131072),
                                 (32, 512), (32, 2048), (32, 8192), (32, 32768)])
def test_decode_sweep_points(B, N):
    """The decode sweep's other points: batch 1 and 32 at 512 .. 128k."""
    case = I.decode_sweep(B, N, device="cuda")
    flag = _flag()
    idx, out, lse = ops.decode_case(case, err_flag=flag)
    torch.cuda.synchronize()
    assert flag.item() == 0
    _check_decode(case, idx, out, lse, sorted({0, B // 2, B - 1}))


def test_packed_long_context_two_loop_full_size():
    """1M-token context on packed fp8_ds_mla pages, SWA 128 + top-k 1024."""
    case = I.packed_long_decode(device="cuda")
    flag = _flag()
    idx, out, lse = ops.decode_case(case, err_flag=flag)
    torch.cuda.synchronize()
    assert flag.item() == 0
    _check_decode(case, idx, out, lse, [0])


def test_uniform_fp8_swa_topk_full_size():
    """Batch 32, 64k context, uniform fp8 pool, shuffled SWA + top-k lists with 10% -1."""
    case = I.uniform_fp8_swa_topk_case(device="cuda")
    flag = _flag()
    out, lse = ops.dsa_sparse_mla_fwd(case.q, case.softmax_scale, case.kv, case.idx, err_flag=flag)
    torch.cuda.synchronize()
    assert flag.item() == 0
    assert (case.idx < 0).sum(dim=1).eq(115).all()
    qn = O.decode_bf16(raw(case.q))
    idx = raw(case.idx)
    pool = pool_np(case.kv)
    for t in range(case.T):
        o, l = O.sparse_mla_one(qn[t], O.gather_valid(pool, idx[t]), case.softmax_scale, 448)
        check_out_lse(out[t].float().cpu().numpy(), lse[t].cpu().numpy(), o, l, "token %d" % t)


# ---------------------------------------------------------------- prefill pipeline

def test_prefill_packed_segments_pipeline():
    """Causal prefill over packed segments (1-token segments included) through
    the three separate entry points: index score -> top-k -> sparse MLA."""
    case = I.prefill_case([1, 1, 700, 2600, 300], k=2048, H=16, device="cuda")
    ind = case.indexer
    maxL = int((case.row_end - case.row_start).max())
    sc = ops.dsa_index_score_prefill(ind["q_idx"], 1, ind["q_scale"], ind["k_idx"],
                                     ind["k_scale"], ind["w"], case.row_start, case.row_end, maxL)
    rl = (case.row_end - case.row_start).contiguous()
    idx, lens = ops.dsa_topk(sc, rl, case.k, maxL, index_base=case.row_start)
    out, lse = ops.dsa_sparse_mla_fwd(case.q, case.softmax_scale, case.kv, idx)
    c = prefill_case_np(case)
    idx_np = idx.cpu().numpy()
    out_np, lse_np = out.float().cpu().numpy(), lse.cpu().numpy()
    r0 = raw(case.row_start)
    for t in [0, 1, 2, 500, 701, 702, 2800, 3301, case.T - 1]:
        r = O.prefill_token(t, c)
        pos = np.where(idx_np[t] >= 0, idx_np[t] - r0[t], -1)
        gset = check_index_sets(pos, r["idx"], r["scores"], case.k)
        if gset is None:
            ref_out, ref_lse = r["out"], r["lse"]
        else:
            ref_out, ref_lse = O.sparse_mla_one(O.decode_bf16(c["q"][t]),
                                                O.gather_valid(c["kv"], gset + r0[t]),
                                                c["softmax_scale"], 512)
        check_out_lse(out_np[t], lse_np[t], ref_out, ref_lse, "token %d" % t)


def test_bounded_wait_gives_up_and_reports():
    """Failure detection: a wait on a barrier nothing completes gives up after
    its limit, reports DSA_DEVERR_TIMEOUT, and the context keeps working."""
    flag, done, waited, limit = ops.selftest_wait_timeout()
    assert flag & ops.DEVERR_TIMEOUT
    assert done == 0 and waited >= limit
    case = I.tiny_decode(device="cuda")
    idx, out, lse = ops.decode_case(case)
    torch.cuda.synchronize()
    assert torch.isfinite(lse).all()
