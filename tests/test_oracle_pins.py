"""Pins for the CPU oracle: hand-worked tables, library routines, brute force
and invariants.  None of these tests needs a GPU."""
import itertools
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle.dsa_oracle as O
from deepseek_sparse_attention_index_gb300 import inputs as I
from tests.helpers import raw, pool_np, decode_case_np

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- dequant

def test_e4m3_hand_table():
    tab = _gold("dequant_hand.json")["e4m3"]
    for code, want in tab.items():
        got = float(O.decode_e4m3(np.array([int(code, 16)], dtype=np.uint8))[0])
        if want == "nan":
            assert math.isnan(got), code
        else:
            assert got == want, (code, got, want)
            assert math.copysign(1.0, got) == math.copysign(1.0, want), code


def test_e4m3_all_codes_match_library_cast():
    codes = np.arange(256, dtype=np.uint8)
    ours = O.decode_e4m3(codes)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    both_nan = np.isnan(ours) & np.isnan(lib)
    assert np.array_equal(np.isnan(ours), np.isnan(lib))
    assert np.array_equal(ours[~both_nan], lib[~both_nan])
    assert np.array_equal(np.signbit(ours[~both_nan]), np.signbit(lib[~both_nan]))


def test_ue8m0_hand():
    for code, want in _gold("dequant_hand.json")["ue8m0"].items():
        assert float(O.decode_ue8m0(np.array([int(code)], dtype=np.uint8))[0]) == want


def test_bf16_hand_and_all_codes():
    for code, want in _gold("dequant_hand.json")["bf16"].items():
        assert float(O.decode_bf16(np.array([int(code, 16)], dtype=np.uint16))[0]) == want
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = O.decode_bf16(codes)
    lib = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    ok = ~np.isnan(lib)
    assert np.array_equal(np.isnan(ours), np.isnan(lib))
    assert np.array_equal(ours[ok], lib[ok])


def test_packed_page_hand():
    g = _gold("dequant_hand.json")["packed_page"]
    block = g["block"]
    page = np.zeros(block * 584, dtype=np.uint8)
    for off, v in g["bytes"].items():
        page[int(off)] = v
    pool = dict(format=O.KV_FP8_DS_MLA, data=page.reshape(1, block, 584), scales=None,
                block=block, d_nope=448, d_rope=64)
    row = O.kv_rows(pool, [g["slot"]])[0]
    assert row.shape == (512,)
    for c, want in g["expect"].items():
        assert row[int(c)] == want, c
    assert np.count_nonzero(row) == 3
    assert not O.kv_rows(pool, [0]).any()


def test_uniform_pool_hand():
    g = _gold("dequant_hand.json")["uniform_pool"]
    D = g["D"]
    data = np.zeros((2, D), dtype=np.uint8)
    for c, v in g["row1_bytes"].items():
        data[1, int(c)] = v
    sc = np.ones((2, D // 64), dtype=np.float32)
    sc[1] = g["row1_scales"]
    pool = dict(format=O.KV_FP8_UNIFORM, data=data, scales=sc, block=1, d_nope=D - 64, d_rope=64)
    row = O.kv_rows(pool, [1])[0]
    for c, want in g["expect_row1"].items():
        assert row[int(c)] == want, c


def test_packed_pool_roundtrip_against_library_decode():
    """Generator's page packer vs the oracle's byte-offset decoder; the
    expected values come from torch's own fp8 / bf16 casts of the parts."""
    block = 4
    n = 8
    g = torch.Generator().manual_seed(5)
    nope = I.to_e4m3_bytes(torch.randn(n, 448, generator=g) * 3)
    exps = torch.randint(120, 135, (n, 7), generator=g).to(torch.uint8)
    rope = torch.randn(n, 64, generator=g).to(torch.bfloat16)
    pages = I.pack_ds_mla_pages(nope, exps, rope, block)
    assert pages.shape == (2, block, 584)
    pool = dict(format=O.KV_FP8_DS_MLA, data=raw(pages), scales=None, block=block,
                d_nope=448, d_rope=64)
    slots = [0, 3, 4, 7, 5]
    got = O.kv_rows(pool, slots)
    nope_v = nope.view(torch.float8_e4m3fn).double()
    scale = torch.exp2(exps.double() - 127.0).repeat_interleave(64, dim=1)
    want = torch.cat([nope_v * scale, rope.double()], dim=1)[slots].numpy()
    assert np.array_equal(got, want)


def test_uniform_pool_roundtrip_against_library_decode():
    pool = I.kv_uniform_fp8_pool(16, seed=3, n=5, device="cpu")
    got = O.kv_rows(pool_np(pool), np.arange(16))
    want = (pool.data.view(torch.float8_e4m3fn).double()
            * pool.scales.double().repeat_interleave(64, dim=1)).numpy()
    assert np.array_equal(got, want)


def test_fp8_row_quantiser_roundtrip():
    x = torch.randn(64, 128, generator=torch.Generator().manual_seed(1))
    q8, s = I.quantize_rows_e4m3(x)
    back = O.decode_e4m3(raw(q8)) * raw(s)[:, None].astype(np.float64)
    # e4m3 keeps 3 mantissa bits: relative error <= 2^-4 above the subnormal range
    err = np.abs(back - x.double().numpy())
    assert np.all(err <= np.maximum(np.abs(x.double().numpy()) * 2.0 ** -4,
                                    raw(s)[:, None] * 2.0 ** -10) + 1e-12)
    assert np.allclose(np.abs(back).max(axis=1), raw(s) * 448.0)


# ---------------------------------------------------------------- index score

def test_index_score_hand_bf16():
    g = _gold("index_score_hand.json")["bf16_case"]
    got = O.index_scores_one(np.array(g["q"]), np.array(g["w"]), np.array(g["k"]))
    assert got.tolist() == g["expect"]


def test_index_score_hand_fp8():
    g = _gold("index_score_hand.json")["fp8_case"]
    q = O.index_values(np.array(g["q_bytes"], dtype=np.uint8), np.array(g["q_scale"]), True)
    k = O.index_values(np.array(g["k_bytes"], dtype=np.uint8), np.array(g["k_scale"]), True)
    got = O.index_scores_one(q, np.array(g["w"]), k)
    assert got.tolist() == g["expect"]


def test_index_score_integer_grid_is_exact_in_fp32():
    """On the integer grid every fp32 partial sum is exact, whatever the order:
    scores in fp64, in fp32 (any order) and in scaled int64 agree exactly."""
    ind = I.indexer_grid_bf16(3, 200, 8, 64, seed=0, device="cpu")
    q = O.decode_bf16(raw(ind["q_idx"]))
    k = O.decode_bf16(raw(ind["k_idx"]))
    w = raw(ind["w"]).astype(np.float64)
    for t in range(3):
        ref = O.index_scores_one(q[t], w[t], k)
        qi = np.rint(q[t] * 8).astype(np.int64)
        ki = np.rint(k * 8).astype(np.int64)
        wi = np.rint(w[t] * 256).astype(np.int64)
        exact = (np.maximum(ki @ qi.T, 0) * wi[None, :]).sum(axis=1)   # units of 2^-14
        assert np.array_equal(ref * 2.0 ** 14, exact.astype(np.float64))
        f32 = (np.maximum(k.astype(np.float32) @ q[t].astype(np.float32).T, 0)
               * w[t].astype(np.float32)).astype(np.float32)
        assert np.array_equal(f32[:, ::-1].sum(axis=1, dtype=np.float32).astype(np.float64), ref)


def test_index_score_invariants():
    rng = np.random.default_rng(0)
    q = rng.standard_normal((6, 16))
    k = rng.standard_normal((30, 16))
    w = rng.standard_normal(6)
    base = O.index_scores_one(q, w, k)
    perm = rng.permutation(6)
    assert np.allclose(O.index_scores_one(q[perm], w[perm], k), base, rtol=1e-13, atol=1e-13)
    assert np.allclose(O.index_scores_one(q, 2.5 * w, k), 2.5 * base, rtol=1e-13, atol=1e-13)
    k2 = k.copy()
    k2[7] = k2[3]
    s2 = O.index_scores_one(q, w, k2)
    assert s2[7] == s2[3]
    # a key anti-aligned with every head contributes nothing
    qa = np.abs(q)
    assert np.all(O.index_scores_one(qa, w, -np.abs(k)) == 0)
    # a single head with w = 1 is ReLU of the plain dot product
    assert np.allclose(O.index_scores_one(q[:1], np.ones(1), k), np.maximum(k @ q[0], 0))


# ---------------------------------------------------------------- top-k

def _brute_topk(s, k):
    L = len(s)
    n = min(L, k)
    good = []
    for sub in itertools.combinations(range(L), n):
        S = set(sub)
        ok = all((s[i] > s[j]) or (s[i] == s[j] and i < j)
                 for i in S for j in range(L) if j not in S)
        if ok:
            good.append(sorted(sub))
    assert len(good) == 1
    return good[0]


def test_topk_brute_force_small():
    rng = np.random.default_rng(1)
    for trial in range(150):
        L = int(rng.integers(1, 11))
        k = int(rng.integers(1, 13))
        s = rng.integers(-3, 4, size=L).astype(np.float64)      # many ties
        got = O.topk_row(s, k)
        n = min(L, k)
        assert (got[n:] == -1).all()
        assert sorted(got[:n].tolist()) == _brute_topk(s, k)


def test_topk_invariants_large():
    rng = np.random.default_rng(2)
    for L, k in [(5000, 2048), (2048, 2048), (100, 2048), (70000, 128)]:
        s = np.round(rng.standard_normal(L) * 50) / 8            # ties present
        got = O.topk_row(s, k)
        n = min(L, k)
        sel = got[:n]
        assert (got[n:] == -1).all() and len(set(sel.tolist())) == n
        mask = np.zeros(L, bool)
        mask[sel] = True
        if n < L:
            lo = s[mask].min()
            assert s[~mask].max() <= lo
            tied_out = np.nonzero((~mask) & (s == lo))[0]
            tied_in = np.nonzero(mask & (s == lo))[0]
            if len(tied_out):
                assert tied_in.max() < tied_out.min()
        else:
            assert sorted(sel.tolist()) == list(range(L))


def test_topk_negative_zero_ties_positive_zero():
    s = np.array([-0.0, 0.0, -0.0, -1.0])
    assert O.topk_row(s, 2).tolist() == [0, 1]


# ---------------------------------------------------------------- sparse MLA

def test_sparse_mla_hand():
    g = _gold("sparse_mla_hand.json")
    pool_rows = np.array(g["pool_rows"])
    for c in g["cases"]:
        idx = np.array(c["idx"])
        rows = pool_rows[idx[idx >= 0]]
        out, lse = O.sparse_mla_one(np.array([c["q"]]), rows, c["scale"], g["Dv"])
        want_lse = -math.inf if c["lse"] == "-inf" else c["lse"]
        assert lse[0] == pytest.approx(want_lse, abs=1e-15) if math.isfinite(want_lse) \
            else lse[0] == want_lse
        assert np.allclose(out[0], c["out"], rtol=0, atol=1e-15)


def _dense_masked(q, pool_rows, sel, scale, Dv):
    """Dense attention over the WHOLE pool with -inf outside the selected set,
    using scipy's logsumexp / softmax."""
    s = scale * (q @ pool_rows.T)
    mask = np.full(pool_rows.shape[0], -np.inf)
    mask[sel] = 0.0
    z = s + mask[None, :]
    lse = scipy.special.logsumexp(z, axis=1)
    p = scipy.special.softmax(z, axis=1)
    return p @ pool_rows[:, :Dv], lse


@pytest.mark.parametrize("fmt", [O.KV_BF16, O.KV_FP8_UNIFORM, O.KV_FP8_DS_MLA])
def test_sparse_mla_matches_dense_masked(fmt):
    rows_n = 512
    if fmt == O.KV_BF16:
        pool = I.kv_bf16_pool(rows_n, 0, 5, "cpu")
        D, Dv = 576, 512
    elif fmt == O.KV_FP8_UNIFORM:
        pool = I.kv_uniform_fp8_pool(rows_n, 0, 5, "cpu")
        D, Dv = 512, 448
    else:
        pool = I.kv_packed_pool(rows_n, 256, 0, 5, "cpu", exp_lo=125, exp_hi=128)
        D, Dv = 512, 448
    pnp = pool_np(pool)
    all_rows = O.kv_rows(pnp, np.arange(rows_n))
    rng = np.random.default_rng(3)
    q = rng.standard_normal((1, 4, D)) * 0.5
    sel = rng.choice(rows_n, 77, replace=False)
    idx = np.concatenate([sel, -np.ones(20, np.int64)])
    rng.shuffle(idx)
    out, lse = O.sparse_mla(q, pnp, idx[None, :], 0.05, Dv)
    dout, dlse = _dense_masked(q[0], all_rows, sel, 0.05, Dv)
    assert np.allclose(out[0], dout, rtol=1e-12, atol=1e-12)
    assert np.allclose(lse[0], dlse, rtol=1e-12, atol=1e-12)


def test_sparse_mla_invariants():
    rng = np.random.default_rng(4)
    rows = rng.standard_normal((40, 8))
    q = rng.standard_normal((3, 8))
    out, lse = O.sparse_mla_one(q, rows, 0.3, 6)
    perm = rng.permutation(40)
    o2, l2 = O.sparse_mla_one(q, rows[perm], 0.3, 6)
    assert np.allclose(out, o2, atol=1e-13) and np.allclose(lse, l2, atol=1e-13)
    # all-equal keys: out is the mean of V
    same = np.tile(rows[:1], (5, 1))
    same[:, :6] = rng.standard_normal((5, 6))
    same[:, 6:] = 1.0
    qz = np.zeros((2, 8))
    qz[:, 6:] = rng.standard_normal((2, 2))
    o3, l3 = O.sparse_mla_one(qz, same, 1.0, 6)
    assert np.allclose(o3, same[:, :6].mean(axis=0)[None, :], atol=1e-13)
    assert np.allclose(l3, (qz[:, 6:].sum(axis=1)) + np.log(5), atol=1e-13)


# ---- attention sinks (a per-head logit in the denominator, no value)

def _sink_case(seed=7, H=4, n=37, D=576, Dv=512):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((H, D))
    rows = rng.standard_normal((n, D))
    sinks = rng.standard_normal(H) * 2.0
    return q, rows, sinks, 1.0 / math.sqrt(192.0), Dv


def test_sink_minus_inf_is_no_sink():
    q, rows, _, sc, Dv = _sink_case()
    out0, lse0 = O.sparse_mla_one(q, rows, sc, Dv)
    out1, lse1 = O.sparse_mla_one(q, rows, sc, Dv, np.full(q.shape[0], -np.inf))
    assert np.allclose(out0, out1, rtol=0, atol=1e-14) and np.allclose(lse0, lse1, rtol=0, atol=1e-14)


def test_sink_equals_an_extra_key_with_zero_value():
    """Brute force: for each head, one more row whose value part (the leading
    Dv columns) is zero and whose RoPE part scores exactly the sink logit gives
    the same result as the sink, through the plain (sink-free) attention."""
    q, rows, sinks, sc, Dv = _sink_case()
    out_s, lse_s = O.sparse_mla_one(q, rows, sc, Dv, sinks)
    for h in range(q.shape[0]):
        qr = q[h, Dv:]
        extra = np.zeros((1, q.shape[1]))
        extra[0, Dv:] = sinks[h] * qr / (sc * qr @ qr)    # sc * q_h . extra = sinks[h]
        out_e, lse_e = O.sparse_mla_one(q[h:h + 1], np.concatenate([rows, extra]), sc, Dv)
        assert np.allclose(out_e[0], out_s[h], rtol=1e-12, atol=1e-13), h
        assert abs(lse_e[0] - lse_s[h]) < 1e-12, h


def test_sink_one_row_closed_form():
    q, rows, sinks, sc, Dv = _sink_case(n=1)
    out, lse = O.sparse_mla_one(q, rows, sc, Dv, sinks)
    s = sc * (q @ rows[0])
    assert np.allclose(lse, np.logaddexp(s, sinks), rtol=0, atol=1e-13)
    weight = 1.0 / (1.0 + np.exp(sinks - s))          # e^s / (e^s + e^sink)
    assert np.allclose(out, weight[:, None] * rows[0, :Dv][None, :], rtol=1e-13, atol=1e-14)


def test_sink_all_masked_row():
    q, rows, sinks, sc, Dv = _sink_case()
    out, lse = O.sparse_mla_one(q, rows[:0], sc, Dv, sinks)
    assert not out.any() and np.array_equal(lse, sinks)


# ---- paged caches (block table)

def _paged_np(shuffle, seed=3):
    case = I.paged_decode(3, [150, 64, 333], page=64, seed=seed, k=128, H=8,
                          idx_kind="bf16_grid", shuffle=shuffle)
    return case, decode_case_np(case)


def test_paged_identity_table_is_the_contiguous_layout():
    case, c = _paged_np(shuffle=False)
    flat = dict(c)
    flat.pop("block_table")
    pages = [(int(L) + 63) // 64 for L in c["seq_lens"]]
    flat["slot_base"] = np.cumsum([0] + [64 * n for n in pages[:-1]])
    for b in range(3):
        r_p, r_c = O.decode_request(b, c), O.decode_request(b, flat)
        assert np.array_equal(r_p["scores"], r_c["scores"]) and np.array_equal(r_p["idx"], r_c["idx"])
        assert np.array_equal(r_p["out"], r_c["out"]) and np.array_equal(r_p["lse"], r_c["lse"])


def test_paged_shuffled_pages_give_the_same_results():
    """The same data with its pages shuffled (and the table following them)
    scores, selects and attends exactly alike."""
    _, c0 = _paged_np(shuffle=False)
    case, c1 = _paged_np(shuffle=True)
    assert not np.array_equal(c0["block_table"], c1["block_table"])
    for b in range(3):
        r0, r1 = O.decode_request(b, c0), O.decode_request(b, c1)
        assert np.array_equal(r0["scores"], r1["scores"]) and np.array_equal(r0["idx"], r1["idx"])
        assert np.array_equal(r0["out"], r1["out"]) and np.array_equal(r0["lse"], r1["lse"])


# ---- backward of the sparse attention

def _bwd_case(seed=11, H=3, n=6, D=12, Dv=8):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((H, D)), rng.standard_normal((n, D)),
            rng.standard_normal((H, Dv)), rng.standard_normal(H), 0.7, Dv)


@pytest.mark.parametrize("with_sinks", [False, True])
def test_sparse_mla_backward_matches_finite_differences(with_sinks):
    """Central differences of L = sum(out * G) against the analytic gradients
    (q, every row entry, every sink)."""
    q, rows, G, sinks, sc, Dv = _bwd_case()
    sk = sinks if with_sinks else None

    def loss(q_, rows_, sk_):
        out, _ = O.sparse_mla_one(q_, rows_, sc, Dv, sk_)
        return float((out * G).sum())

    dq, drows, dsk = O.sparse_mla_bwd_one(q, rows, G, sc, Dv, sk)
    eps = 1e-6
    for arr, grad in ((q, dq), (rows, drows)):
        num = np.zeros_like(arr)
        for i in np.ndindex(arr.shape):
            a0 = arr[i]
            arr[i] = a0 + eps
            lp = loss(q, rows, sk)
            arr[i] = a0 - eps
            lm = loss(q, rows, sk)
            arr[i] = a0
            num[i] = (lp - lm) / (2 * eps)
        assert np.allclose(grad, num, rtol=1e-6, atol=1e-8)
    if with_sinks:
        for h in range(len(sinks)):
            s0 = sinks[h]
            sinks[h] = s0 + eps
            lp = loss(q, rows, sinks)
            sinks[h] = s0 - eps
            lm = loss(q, rows, sinks)
            sinks[h] = s0
            assert abs(dsk[h] - (lp - lm) / (2 * eps)) < 1e-7
    else:
        assert not dsk.any()


def test_sparse_mla_backward_scatter_adds_shared_rows():
    """Two tokens selecting the same slot (and -1 entries) add their row
    gradients into that slot; a slot nobody selects gets zero."""
    pool = I.kv_bf16_pool(16, 1, 5, "cpu")
    pn = pool_np(pool)
    rng = np.random.default_rng(3)
    q = rng.standard_normal((2, 4, 576)) * 0.1
    dout = rng.standard_normal((2, 4, 512))
    idx = np.array([[3, 7, -1, 9], [7, 3, 12, -1]])
    dq, dkv, _ = O.sparse_mla_bwd(q, pn, idx, dout, 0.05, 512)
    for t in range(2):
        sl = idx[t][idx[t] >= 0]
        dq1, dr1, _ = O.sparse_mla_bwd_one(q[t], O.kv_rows(pn, sl), dout[t], 0.05, 512)
        assert np.allclose(dq[t], dq1)
    r0 = O.sparse_mla_bwd_one(q[0], O.kv_rows(pn, [3, 7, 9]), dout[0], 0.05, 512)[1]
    r1 = O.sparse_mla_bwd_one(q[1], O.kv_rows(pn, [7, 3, 12]), dout[1], 0.05, 512)[1]
    assert np.allclose(dkv[7], r0[1] + r1[0]) and np.allclose(dkv[3], r0[0] + r1[1])
    assert not dkv[0].any() and not dkv[15].any()


def test_split_combine_equals_whole():
    rng = np.random.default_rng(5)
    rows = rng.standard_normal((100, 16)) * 2
    q = rng.standard_normal((4, 16))
    out, lse = O.sparse_mla_one(q, rows, 0.7, 12)
    parts = [rows[:13], rows[13:13], rows[13:70], rows[70:]]
    po, pl = zip(*[O.sparse_mla_one(q, p, 0.7, 12) for p in parts])
    for h in range(4):
        o, l = O.combine_splits(np.stack([x[h] for x in po]), np.array([x[h] for x in pl]))
        assert np.allclose(o, out[h], atol=1e-13) and abs(l - lse[h]) < 1e-13


def test_two_loop_equals_concatenated_list():
    rng = np.random.default_rng(6)
    a = I.kv_packed_pool(256, 256, 1, 5, "cpu", exp_lo=126, exp_hi=128)
    b = I.kv_packed_pool(512, 256, 2, 6, "cpu", exp_lo=126, exp_hi=128)
    pa, pb = pool_np(a), pool_np(b)
    q = rng.standard_normal((2, 4, 512))
    ia = rng.choice(256, (2, 30)).astype(np.int64)
    ib = rng.choice(512, (2, 50)).astype(np.int64)
    ib[:, ::7] = -1
    out, lse = O.sparse_mla(q, pa, ia, 0.04, 448, pb, ib)
    for t in range(2):
        rows = np.concatenate([O.kv_rows(pa, ia[t]), O.kv_rows(pb, ib[t][ib[t] >= 0])])
        o, l = O.sparse_mla_one(q[t], rows, 0.04, 448)
        assert np.allclose(out[t], o, atol=1e-13) and np.allclose(lse[t], l, atol=1e-13)


# ---------------------------------------------------------------- decode

def test_decode_k_at_least_context_is_full_attention():
    """With k >= context the step attends to every context row: compare with
    dense attention over rows [0, L) through scipy."""
    case = I.decode_case("t", 2, [300, 41], 8, 64, "bf16_grid", 512, 4, I.KV_BF16, device="cpu")
    c = decode_case_np(case)
    for b in range(2):
        r = O.decode_request(b, c)
        L = int(c["seq_lens"][b])
        base = int(c["slot_base"][b])
        assert sorted(r["idx"][:L].tolist()) == list(range(L)) and (r["idx"][L:] == -1).all()
        rows = O.kv_rows(c["kv"], base + np.arange(L))
        dout, dlse = _dense_masked(O.decode_bf16(c["q"][b]), rows, np.arange(L),
                                   c["softmax_scale"], 512)
        assert np.allclose(r["out"], dout, atol=1e-12) and np.allclose(r["lse"], dlse, atol=1e-12)


def test_decode_composition_tiny():
    case = I.tiny_decode()
    c = decode_case_np(case)
    r = O.decode_request(0, c)
    assert r["scores"].shape == (512,)
    assert (r["idx"] >= 0).all() and len(set(r["idx"].tolist())) == 128
    assert r["idx"].tolist() == O.topk_row(r["scores"], 128).tolist()
    rows = O.kv_rows(c["kv"], r["idx"])
    o, l = O.sparse_mla_one(O.decode_bf16(c["q"][0]), rows, c["softmax_scale"], 512)
    assert np.array_equal(o, r["out"]) and np.array_equal(l, r["lse"])
