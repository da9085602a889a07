"""The C-ABI library builds, loads and exports every function include/dsa.h
declares; host-side argument checks reject bad calls before any launch.
No GPU is needed: nothing here reaches a kernel."""
import ctypes
import os

import pytest

from deepseek_sparse_attention_index_gb300 import build as B
from deepseek_sparse_attention_index_gb300 import ops


@pytest.fixture(scope="module")
def lib():
    B.build()
    return ops.load()


def test_header_declares_the_boundary():
    names = ops.header_functions()
    for n in ["dsa_index_score", "dsa_topk", "dsa_sparse_mla_fwd", "dsa_decode",
              "dsa_topk_workspace_size", "dsa_sparse_mla_workspace_size",
              "dsa_decode_workspace_size", "dsa_status_string", "dsa_abi_version",
              "dsa_sparse_mla_fwd_ex", "dsa_decode_ex", "dsa_decode_paged", "dsa_decode_host",
              "dsa_decode_host_workspace_size", "dsa_sparse_mla_bwd", "dsa_index_score_prefill"]:
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in ops.header_functions():
        assert hasattr(lib, n), n
        assert n in ops._SIGS, "binding lacks a signature for " + n


def test_version_and_status_strings(lib):
    assert lib.dsa_abi_version() == 1
    for code in range(5):
        assert lib.dsa_status_string(code)
    assert lib.dsa_status_string(99) == b"unknown status"


FAKE = ctypes.c_void_p(0x10000)  # 16-byte aligned, never dereferenced


def test_topk_rejects_bad_arguments(lib):
    # k out of range
    assert lib.dsa_topk(FAKE, 8, FAKE, 1, 8, 0, None, FAKE, None, FAKE, 1 << 20, None,
                        None) == 2
    assert lib.dsa_topk(FAKE, 8, FAKE, 1, 8, ops.MAX_TOPK + 1, None, FAKE, None, FAKE, 1 << 20,
                        None, None) == 2
    # ld smaller than max_len
    assert lib.dsa_topk(FAKE, 4, FAKE, 1, 8, 2, None, FAKE, None, FAKE, 1 << 20, None, None) == 1
    # workspace too small
    need = lib.dsa_topk_workspace_size(3, 100, 16)
    assert need > 0
    assert lib.dsa_topk(FAKE, 100, FAKE, 3, 100, 16, None, FAKE, None, FAKE, need - 1, None,
                        None) == 3
    # T = 0 is a no-op
    assert lib.dsa_topk(None, 0, None, 0, 0, 4, None, None, None, None, 0, None, None) == 0


def _pool(fmt, rows=16, block=1, d_nope=512, scales=True):
    p = ops.DsaKvPool()
    p.data = FAKE.value
    p.scales = FAKE.value if scales else None
    p.rows = rows
    p.format = fmt
    p.block = block
    p.d_nope = d_nope
    p.d_rope = 64
    return p


def _mla(lib, pool, D=576, Dv=512, H=8, k=4, idx=FAKE, ws_bytes=1 << 30, scale=0.1, q=FAKE):
    return lib.dsa_sparse_mla_fwd(q, 2, H, D, Dv, scale, ctypes.byref(pool), idx, k, None, None,
                                  0, FAKE, FAKE, FAKE, ws_bytes, None, None)


def test_sparse_mla_rejects_bad_arguments(lib):
    assert _mla(lib, _pool(0, d_nope=512), D=512, Dv=448) == 2        # bf16 pool must be 576
    assert _mla(lib, _pool(0, d_nope=512), D=576, Dv=448) == 2        # (D, Dv) pair
    assert _mla(lib, _pool(0, d_nope=512), H=0) == 2
    assert _mla(lib, _pool(0, d_nope=512), H=ops.MAX_TOPK) == 2
    assert _mla(lib, _pool(1, d_nope=448, scales=False), D=512, Dv=448) == 1  # no scales
    assert _mla(lib, _pool(2, rows=512, block=255, d_nope=448), D=512, Dv=448) == 2  # odd block
    assert _mla(lib, _pool(2, rows=500, block=256, d_nope=448), D=512, Dv=448) == 1  # rows % block
    assert _mla(lib, _pool(0, d_nope=512), idx=None) == 1
    p = _pool(0, d_nope=512)
    p.data = 0x10004                                                      # misaligned pool
    assert _mla(lib, p) == 1
    need = lib.dsa_sparse_mla_workspace_size(2, 8, 512, 4, 0)
    if need:
        assert _mla(lib, _pool(0, d_nope=512), ws_bytes=need - 1) == 3
    # the softmax scale must be positive and finite
    for bad in (0.0, -0.1, float("nan"), float("inf")):
        assert _mla(lib, _pool(0, d_nope=512), scale=bad) == 1, bad
    # q must start on a 16-byte boundary
    assert _mla(lib, _pool(0, d_nope=512), q=ctypes.c_void_p(FAKE.value + 2)) == 1


@pytest.mark.parametrize("entry", ["dsa_index_score", "dsa_index_score_prefill"])
def test_index_score_rejects_bad_arguments(lib, entry):
    def call(idx_dtype=1, H_I=64, d=128, q_scale=FAKE, ld=128, max_len=100):
        return getattr(lib, entry)(FAKE, idx_dtype, q_scale, FAKE, FAKE, 1000, FAKE, FAKE, FAKE,
                                   8, H_I, d, max_len, FAKE, ld, None, None)
    assert call(H_I=65) == 2
    assert call(H_I=12) == 2
    assert call(d=64) == 2           # fp8 needs d = 128
    assert call(idx_dtype=7) == 2
    assert call(q_scale=None) == 1   # fp8 needs scales
    assert call(ld=50) == 1          # ld < max_len


def test_workspace_sizes_grow_with_the_problem(lib):
    a = lib.dsa_decode_workspace_size(1, 1 << 14, 2048, 64, 512, 0)
    b = lib.dsa_decode_workspace_size(32, 1 << 17, 2048, 64, 512, 0)
    assert 0 < a < b
    assert b >= 32 * (1 << 17) * 4   # the score rows live in the workspace


def _opts(rows_per_request=0, lse_log2=0):
    o = ops.DsaAttnOpts()
    o.sinks = None
    o.lse_log2 = lse_log2
    o.rows_per_request = rows_per_request
    return o


def test_rows_per_request_is_a_decode_option_only(lib):
    st = lib.dsa_sparse_mla_fwd_ex(FAKE, 2, 8, 576, 512, 0.1, ctypes.byref(_pool(0, d_nope=512)),
                                   FAKE, 4, None, None, 0, FAKE, FAKE, FAKE, 1 << 30, None,
                                   ctypes.byref(_opts(rows_per_request=2)), None)
    assert st == 1


def test_decode_rows_per_request_checks(lib):
    def call(rpr, B=4, idx_dtype=1, H_I=64, d=128):
        return lib.dsa_decode_ex(FAKE, idx_dtype, FAKE, FAKE, FAKE, 1 << 20, FAKE, H_I, d, B,
                                 FAKE, FAKE, 1000, 64, FAKE, 8, 576, 512, 0.1,
                                 ctypes.byref(_pool(0, rows=1 << 20, d_nope=512)), None, None, 0,
                                 None, FAKE, FAKE, FAKE, 1 << 34, None,
                                 ctypes.byref(_opts(rows_per_request=rpr)), None)
    assert call(3) == 2                  # pairs only
    assert call(-1) == 2
    assert call(2, B=3) == 1             # rows come in pairs
    assert call(2, H_I=128) == 2         # two rows of at most 64 heads
    assert call(2, idx_dtype=0, d=128) == 2   # bf16 indexer: d = 64 only


def test_decode_paged_rejects_bad_arguments(lib):
    def call(page=64, max_pages=16, max_len=1000, bt=FAKE, k=64, opts=None):
        return lib.dsa_decode_paged(FAKE, 1, FAKE, FAKE, FAKE, 1 << 20, FAKE, 64, 128, 2, FAKE, bt,
                                    max_pages, page, max_len, k, FAKE, 8, 576, 512, 0.1,
                                    ctypes.byref(_pool(0, rows=1 << 20, d_nope=512)), None, None, 0,
                                    None, FAKE, FAKE, FAKE, 1 << 34, None,
                                    None if opts is None else ctypes.byref(opts), None)
    assert call(page=50) == 2           # pages are multiples of 64 slots
    assert call(page=0) == 2
    assert call(max_pages=3) == 1       # 3 x 64 < max_seq_len
    assert call(bt=None) == 1           # no block table
    assert call(k=0) == 2
    assert call(opts=_opts(rows_per_request=2)) == 1


def test_sparse_mla_backward_rejects_bad_arguments(lib):
    def call(pool=None, D=576, Dv=512, dq=FAKE, T=2, k=4):
        pool = pool if pool is not None else _pool(0, d_nope=512)
        return lib.dsa_sparse_mla_bwd(FAKE, T, 8, D, Dv, 0.1, ctypes.byref(pool), FAKE, k, FAKE,
                                      FAKE, None, dq, FAKE, None, None, None)
    assert call(pool=_pool(1, d_nope=448), D=512, Dv=448) == 2   # bf16 pools only
    assert call(D=512) == 2
    assert call(dq=None) == 1
    assert call(k=0) == 1
    assert call(T=0) == 0


def test_decode_host_rejects_bad_arguments(lib):
    need = lib.dsa_decode_host_workspace_size(2, 1000, 64, 64, 128, 1, 8, 576, 512, 0)
    assert need > lib.dsa_decode_workspace_size(2, 1000, 64, 8, 512, 0)

    def call(h_q=FAKE, ws_bytes=need, k=64):
        return lib.dsa_decode_host(FAKE, 1, FAKE, FAKE, FAKE, 1 << 20, FAKE, 64, 128, 2, FAKE,
                                   FAKE, 1000, k, h_q, 8, 576, 512, 0.1,
                                   ctypes.byref(_pool(0, rows=1 << 20, d_nope=512)), None, None, 0,
                                   None, FAKE, FAKE, FAKE, ws_bytes, None, None)
    assert call(h_q=None) == 1
    assert call(ws_bytes=need - 1) == 3
    assert call(k=ops.MAX_TOPK + 1) == 2


def test_decode_graph_host_rejections(lib):
    """No graph is made: a NULL out-handle or an empty batch is rejected before
    any CUDA call; launching or destroying a NULL handle is harmless."""
    pool = _pool(0, d_nope=512)
    h = ctypes.c_void_p(1234)
    def create(B=2, out=ctypes.byref(h)):
        return lib.dsa_decode_graph_create(FAKE, 1, FAKE, FAKE, FAKE, 1000, FAKE, 64, 128, B, FAKE,
                                           FAKE, 4096, 2048, FAKE, 64, 576, 512, 0.1,
                                           ctypes.byref(pool), None, None, 0, None, FAKE, FAKE,
                                           FAKE, 1 << 30, None, out)
    assert create(out=None) == 1
    assert create(B=0) == 1 and h.value is None
    assert lib.dsa_decode_graph_launch(None, None) == 1
    lib.dsa_decode_graph_destroy(None)


def test_header_is_plain_c(tmp_path):
    """include/dsa.h is a C ABI: it compiles as strict C99 with only the C
    standard headers (no CUDA or C++ types in the signatures)."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not installed")
    src = tmp_path / "use_header.c"
    src.write_text('#include "dsa.h"\n'
                   "int main(void) { dsa_decode_graph g = 0; (void)g; return dsa_abi_version() ? 0 : 1; }\n")
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", inc,
                        "-c", str(src), "-o", str(tmp_path / "use_header.o")],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
