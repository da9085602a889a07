"""dsa_decode_host: the fused decode step with the step's inputs and outputs in
host memory.  It runs the kernels of dsa_decode on device copies of the
inputs, so its results must equal dsa_decode's bit for bit; dsa_decode itself
is checked against the oracle in test_gpu_parity.py.  One case here is also
checked against the oracle directly."""
import pytest
import torch

from deepseek_sparse_attention_index_gb300 import build as B
from deepseek_sparse_attention_index_gb300 import inputs as I
from deepseek_sparse_attention_index_gb300 import ops
from tests.test_gpu_parity import _check_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    B.build()
    ops.load()


def _pin(t):
    return None if t is None else t.detach().cpu().contiguous().pin_memory()


def _host_inputs(case):
    ind = case.indexer
    return dict(q_idx=_pin(ind["q_idx"]), q_scale=_pin(ind["q_scale"]), w=_pin(ind["w"]),
                seq_lens=_pin(case.seq_lens), slot_base=_pin(case.slot_base), q=_pin(case.q),
                idx_swa=_pin(case.idx_swa))


def _run_host(case, h, **kw):
    ind = case.indexer
    return ops.dsa_decode_host(h["q_idx"], ind["idx_dtype"], h["q_scale"], ind["k_idx"],
                               ind["k_scale"], h["w"], h["seq_lens"], h["slot_base"],
                               case.max_seq_len, case.k, h["q"], case.softmax_scale, case.kv,
                               kv_swa=case.kv_swa, idx_swa=h["idx_swa"], **kw)


def _same(host, dev):
    assert torch.equal(host, dev.cpu()), "host-buffer decode differs from the device call"


@pytest.mark.parametrize("name,make", [
    ("fp8_ragged", lambda: I.decode_case("host_fp8", 5, [1, 300, 2048, 2049, 10000], 64, 128,
                                         "fp8", 2048, 64, I.KV_BF16, device="cuda")),
    ("bf16_grid", lambda: I.tiny_decode(device="cuda")),
    ("packed_two_loop", lambda: I.decode_case("host_packed", 3, [5000, 20000, 70000], 64, 128,
                                              "fp8", 1024, 64, I.KV_FP8_DS_MLA, device="cuda",
                                              swa=128)),
    ("uniform_fp8", lambda: I.decode_case("host_uniform", 4, [700, 4096, 9000, 30000], 64, 128,
                                          "fp8", 2048, 64, I.KV_FP8_UNIFORM, device="cuda")),
])
def test_decode_host_equals_device_call(name, make):
    case = make()
    idx_d, out_d, lse_d = ops.decode_case(case)
    h = _host_inputs(case)
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx_h, out_h, lse_h = _run_host(case, h, err_flag=flag)
    torch.cuda.synchronize()
    assert flag.item() == 0
    for t in (idx_h, out_h, lse_h):
        assert not t.is_cuda
    _same(idx_h, idx_d)
    _same(out_h, out_d)
    _same(lse_h, lse_d)


def test_decode_host_pageable_buffers_equal_pinned():
    """Pinned host buffers are moved by copy kernels, pageable ones by the copy
    engines: the same results either way (odd sizes leave byte tails)."""
    case = I.decode_case("host_pageable", 3, [700, 5000, 20001], 64, 128, "fp8", 2048, 64,
                         I.KV_BF16, device="cuda")
    h = _host_inputs(case)
    pageable = {k: (None if v is None else v.clone()) for k, v in h.items()}
    assert all(v is None or not v.is_pinned() for v in pageable.values())
    a = _run_host(case, h)
    b = _run_host(case, pageable, idx_out=torch.empty((3, case.k), dtype=torch.int32),
                  out=torch.empty((3, case.H, case.Dv), dtype=torch.bfloat16),
                  lse=torch.empty((3, case.H), dtype=torch.float32))
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_decode_host_against_oracle():
    case = I.decode_case("host_oracle", 3, [129, 2500, 6000], 64, 128, "fp8", 2048, 64, I.KV_BF16,
                         device="cuda")
    idx_h, out_h, lse_h = _run_host(case, _host_inputs(case))
    torch.cuda.synchronize()
    _check_decode(case, idx_h, out_h, lse_h, range(case.B))


def test_decode_host_back_to_back_steps_share_one_workspace():
    """Two steps enqueued without a host synchronisation between them, on one
    workspace and one stream: the second step's input copies must not land
    before the first step has finished reading its staged inputs."""
    a = I.decode_case("host_a", 4, [3000, 9000, 20000, 40000], 64, 128, "fp8", 2048, 64,
                      I.KV_BF16, device="cuda", seed=1)
    b = I.decode_case("host_b", 4, [3000, 9000, 20000, 40000], 64, 128, "fp8", 2048, 64,
                      I.KV_BF16, device="cuda", seed=2)
    ref_a = ops.decode_case(a)
    ref_b = ops.decode_case(b)
    ind = a.indexer
    need = ops.dsa_decode_host_workspace_size(a.B, a.max_seq_len, a.k, a.H_I, a.d_idx,
                                              ind["idx_dtype"], a.H, a.D, a.Dv)
    ws = ops.workspace(need, "cuda")
    # the second step's indexer state is b's; both steps read their own caches
    got_a = _run_host(a, _host_inputs(a), ws=ws)
    got_b = _run_host(b, _host_inputs(b), ws=ws)
    torch.cuda.synchronize()
    for got, ref in ((got_a, ref_a), (got_b, ref_b)):
        for x, y in zip(got, ref):
            _same(x, y)


def test_decode_host_rejects_device_tensors_and_small_workspace():
    case = I.tiny_decode(device="cuda")
    h = _host_inputs(case)
    bad = dict(h)
    bad["q"] = case.q          # a CUDA tensor where a host buffer is expected
    with pytest.raises(ValueError):
        _run_host(case, bad)
    with pytest.raises(ops.DsaError):
        _run_host(case, h, ws=ops.workspace(16, "cuda"))


# ---------------------------------------------------------------- dsa_decode_graph

def _graph(case, h, **kw):
    ind = case.indexer
    return ops.DecodeGraph(h["q_idx"], ind["idx_dtype"], h["q_scale"], ind["k_idx"],
                           ind["k_scale"], h["w"], h["seq_lens"], h["slot_base"],
                           case.max_seq_len, case.k, h["q"], case.softmax_scale, case.kv,
                           kv_swa=case.kv_swa, idx_swa=h["idx_swa"], **kw)


@pytest.mark.parametrize("name,make", [
    ("fp8_ragged", lambda: I.decode_case("graph_fp8", 5, [1, 300, 2048, 2049, 10000], 64, 128,
                                         "fp8", 2048, 64, I.KV_BF16, device="cuda")),
    ("packed_two_loop", lambda: I.decode_case("graph_packed", 3, [5000, 20000, 70000], 64, 128,
                                              "fp8", 1024, 64, I.KV_FP8_DS_MLA, device="cuda",
                                              swa=128)),
])
def test_decode_graph_replays_equal_direct_calls(name, make):
    """A captured step, launched twice: first on the case's inputs, then on
    inputs rewritten in place in the same pinned buffers (other queries,
    shorter contexts, the same caches).  Each launch equals dsa_decode on the
    same inputs bit for bit."""
    import dataclasses
    case = make()
    h = _host_inputs(case)
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = _graph(case, h, err_flag=flag)
    try:
        for step in range(2):
            if step == 1:
                # step 2: new queries and weights, every context shortened
                ind = dict(case.indexer)
                gen = torch.Generator(device="cuda").manual_seed(7)
                ind["w"] = (torch.randn(ind["w"].shape, generator=gen, device="cuda") / 8).contiguous()
                q = I.to_bf16(torch.randn(case.q.shape, generator=gen, device="cuda")).contiguous()
                seq = (case.seq_lens - torch.clamp(case.seq_lens // 3, max=500)).clamp(min=1)
                case = dataclasses.replace(case, indexer=ind, q=q, seq_lens=seq.to(torch.int32).contiguous())
                for key, src in (("w", ind["w"]), ("q", q), ("seq_lens", case.seq_lens)):
                    h[key].copy_(src.cpu())
            got = g.launch()
            torch.cuda.synchronize()
            ref = ops.decode_case(case)
            torch.cuda.synchronize()
            for x, y in zip(got, ref):
                _same(x, y)
        assert flag.item() == 0
    finally:
        g.close()


def test_decode_graph_rejects_pageable_buffers_and_bad_shapes():
    case = I.tiny_decode(device="cuda")
    h = _host_inputs(case)
    bad = dict(h)
    bad["q"] = case.q.cpu()            # pageable: the graph's copies need pinned memory
    with pytest.raises(ValueError):
        _graph(case, bad)
    with pytest.raises(ops.DsaError):
        _graph(case, h, ws=ops.workspace(16, "cuda"))
