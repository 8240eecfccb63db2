"""The C-ABI library without a GPU: it builds, loads, exports every symbol of
include/nbx.h, and refuses bad arguments on the host before any CUDA call."""

import ctypes
import json
import os
import re

import pytest

import paged_split_kv_append_gb300 as nbx

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nbx.h")

NULL = None
FAKE = ctypes.c_void_p(0x10000)          # a 16-byte aligned address that is never dereferenced
FAKE_ODD = ctypes.c_void_p(0x10008)


@pytest.fixture(scope="module")
def lib():
    nbx.build()
    return nbx.lib()


def declared_symbols():
    text = open(HEADER).read()
    return re.findall(r"NBX_API\s+[\w\s\*]+?\b(nbx_\w+)\s*\(", text)


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for s in ("nbx_paged_kv_append", "nbx_paged_decode_workspace_bytes", "nbx_paged_decode_attn",
              "nbx_paged_decode_merge", "nbx_status_string", "nbx_abi_version", "nbx_set_decode_grid_limit",
              "nbx_paged_decode_step", "nbx_decode_attn_contiguous"):
        assert s in syms


def test_library_exports_every_declared_symbol(lib):
    for s in declared_symbols():
        assert hasattr(lib, s), s


def test_status_strings(lib):
    assert nbx.nbx_status_string(0) == "ok"
    for code in range(-1, -9, -1):
        assert nbx.nbx_status_string(code) != "unknown status"
    assert lib.nbx_abi_version() == 100


def _append(lib, **kw):
    a = dict(new_k=FAKE, new_v=FAKE, new_dtype=0, n_tok=4, h_kv=2, d=64, k_pool=FAKE, v_pool=FAKE, pool_dtype=1,
             num_pages=8, page_tokens=16, slots=FAKE, k_scale=1.0, v_scale=1.0, status=NULL, stream=NULL)
    a.update(kw)
    return lib.nbx_paged_kv_append(a["new_k"], a["new_v"], a["new_dtype"], a["n_tok"], a["h_kv"], a["d"],
                                   a["k_pool"], a["v_pool"], a["pool_dtype"], a["num_pages"], a["page_tokens"],
                                   a["slots"], a["k_scale"], a["v_scale"], a["status"], a["stream"])


def test_append_host_checks(lib):
    assert _append(lib, n_tok=0) == 0                        # nothing to write: no launch
    assert _append(lib, new_k=NULL) == -1
    assert _append(lib, slots=NULL) == -1
    assert _append(lib, d=72) == -2
    assert _append(lib, h_kv=0) == -2
    assert _append(lib, n_tok=-1) == -2
    assert _append(lib, new_dtype=2) == -3                   # e4m3 input is not taken
    assert _append(lib, pool_dtype=7) == -3
    assert _append(lib, k_pool=FAKE_ODD) == -7
    assert _append(lib, v_scale=0.0) == -8
    assert _append(lib, k_scale=float("nan")) == -8


def _decode(lib, **kw):
    a = dict(q=FAKE, q_dtype=1, batch=2, rows=1, h_q=8, d=128, k_pool=FAKE, v_pool=FAKE, pool_dtype=1,
             num_pages=100, h_kv=2, page_tokens=16, bt=FAKE, max_pages=10, lens=FAKE, max_seq_len=160,
             scale=0.1, k_scale=1.0, v_scale=1.0, out=FAKE, ws=FAKE, ws_bytes=1 << 30, status=NULL, stream=NULL)
    a.update(kw)
    return lib.nbx_paged_decode_attn(a["q"], a["q_dtype"], a["batch"], a["rows"], a["h_q"], a["d"], a["k_pool"],
                                     a["v_pool"], a["pool_dtype"], a["num_pages"], a["h_kv"], a["page_tokens"],
                                     a["bt"], a["max_pages"], a["lens"], a["max_seq_len"], a["scale"],
                                     a["k_scale"], a["v_scale"], a["out"], a["ws"], a["ws_bytes"], a["status"],
                                     a["stream"])


def test_decode_host_checks(lib):
    assert _decode(lib, batch=0) == 0                        # empty batch: no launch
    assert _decode(lib, h_q=6, h_kv=4) == -2                 # h_q % h_kv
    assert _decode(lib, d=96) == -2
    assert _decode(lib, rows=0) == -2
    assert _decode(lib, max_seq_len=161) == -2               # more positions than the table holds
    assert _decode(lib, page_tokens=24, max_seq_len=100) == -4   # a tile would straddle two pages
    assert _decode(lib, q_dtype=2) == -3
    assert _decode(lib, pool_dtype=5) == -3
    assert _decode(lib, scale=float("inf")) == -8
    assert _decode(lib, v_scale=-1.0) == -8
    assert _decode(lib, bt=NULL) == -1
    assert _decode(lib, ws=NULL) == -1
    assert _decode(lib, out=FAKE_ODD) == -7
    assert _decode(lib, ws=ctypes.c_void_p(0x10010)) == -7   # workspace must be 256-byte aligned
    need = lib.nbx_paged_decode_workspace_bytes(2, 1, 8, 2, 128, 160)
    assert _decode(lib, ws_bytes=need - 1) == -5


def _step(lib, **kw):
    a = dict(q=FAKE, q_dtype=1, batch=2, rows=1, h_q=8, d=128, nk=FAKE, nv=FAKE, new_dtype=0, k_pool=FAKE,
             v_pool=FAKE, pool_dtype=1, num_pages=100, h_kv=2, page_tokens=16, bt=FAKE, max_pages=10, lens=FAKE,
             max_seq_len=160, scale=0.1, k_scale=1.0, v_scale=1.0, out=FAKE, ws=FAKE, ws_bytes=1 << 30,
             status=NULL, stream=NULL)
    a.update(kw)
    return lib.nbx_paged_decode_step(a["q"], a["q_dtype"], a["batch"], a["rows"], a["h_q"], a["d"], a["nk"],
                                     a["nv"], a["new_dtype"], a["k_pool"], a["v_pool"], a["pool_dtype"],
                                     a["num_pages"], a["h_kv"], a["page_tokens"], a["bt"], a["max_pages"],
                                     a["lens"], a["max_seq_len"], a["scale"], a["k_scale"], a["v_scale"], a["out"],
                                     a["ws"], a["ws_bytes"], a["status"], a["stream"])


def test_step_host_checks(lib):
    # every refusal happens before the step's append is launched
    assert _step(lib, batch=0) == 0
    assert _step(lib, h_q=6, h_kv=4) == -2
    assert _step(lib, max_seq_len=161) == -2
    assert _step(lib, page_tokens=24, max_seq_len=100) == -4
    assert _step(lib, new_dtype=2) == -3                     # new keys are fp32 or bf16
    assert _step(lib, pool_dtype=7) == -3
    assert _step(lib, k_scale=0.0) == -8
    assert _step(lib, nk=NULL) == -1
    assert _step(lib, lens=NULL) == -1
    assert _step(lib, bt=NULL) == -1
    assert _step(lib, nv=FAKE_ODD) == -7
    need = lib.nbx_paged_decode_workspace_bytes(2, 1, 8, 2, 128, 160)
    assert _step(lib, ws_bytes=need - 1) == -5


def _contig(lib, **kw):
    a = dict(q=FAKE, q_dtype=1, batch=2, rows=1, h_q=8, d=128, k=FAKE, v=FAKE, dtype=1, h_kv=2, capacity=160,
             lens=FAKE, max_seq_len=160, scale=0.1, k_scale=1.0, v_scale=1.0, out=FAKE, ws=FAKE, ws_bytes=1 << 30,
             status=NULL, stream=NULL)
    a.update(kw)
    return lib.nbx_decode_attn_contiguous(a["q"], a["q_dtype"], a["batch"], a["rows"], a["h_q"], a["d"], a["k"],
                                          a["v"], a["dtype"], a["h_kv"], a["capacity"], a["lens"],
                                          a["max_seq_len"], a["scale"], a["k_scale"], a["v_scale"], a["out"],
                                          a["ws"], a["ws_bytes"], a["status"], a["stream"])


def test_contiguous_host_checks(lib):
    assert _contig(lib, batch=0) == 0
    assert _contig(lib, capacity=0) == -2
    assert _contig(lib, max_seq_len=161) == -2               # more positions than the cache holds
    assert _contig(lib, capacity=40, max_seq_len=40) == -4   # capacity: whole 16-position tiles
    assert _contig(lib, dtype=9) == -3
    assert _contig(lib, k=NULL) == -1
    assert _contig(lib, lens=NULL) == -1
    assert _contig(lib, out=FAKE_ODD) == -7
    need = lib.nbx_paged_decode_workspace_bytes_for(1, 1, 2, 1, 8, 2, 128, 160, 160)
    assert _contig(lib, ws_bytes=need - 1) == -5


def test_workspace_bytes(lib):
    f = lib.nbx_paged_decode_workspace_bytes
    assert f(2, 1, 8, 3, 128, 100) == 0                      # invalid sizes -> 0
    small = f(32, 1, 32, 8, 128, 8192)
    big = f(32, 1, 32, 8, 128, 131072)
    assert 0 < small < big
    # the fp32 partials dominate: batch * rows * h_q * splits(max_seq_len) * (d + 2) floats
    assert big >= 32 * 32 * 64 * 130 * 4
    assert small >= 32 * 32 * 32 * 130 * 4


def test_merge_host_checks(lib):
    f = lib.nbx_paged_decode_merge
    assert f(FAKE, FAKE, FAKE, 0, 4, 64, FAKE, NULL) == 0
    assert f(FAKE, FAKE, FAKE, 3, 0, 64, FAKE, NULL) == -2
    assert f(FAKE, FAKE, FAKE, 3, 4, 0, FAKE, NULL) == -2
    assert f(NULL, FAKE, FAKE, 3, 4, 64, FAKE, NULL) == -1


def test_binding_fails_loudly_without_the_library(monkeypatch, tmp_path):
    monkeypatch.setattr(nbx, "_lib", None)
    monkeypatch.setattr(nbx._build, "LIB", str(tmp_path / "missing" / "libnbx.so"))
    with pytest.raises(nbx.NbxLibraryMissing):
        nbx.lib()


def test_partial_kernel_choice(lib):
    # rows x group >= 64 with bf16 q and pools, d 128/256, 64-position pages: tensor cores
    assert nbx.nbx_paged_decode_partial_kernel(nbx.NBX_BF16, nbx.NBX_BF16, 16, 24, 4, 256, 1000, 64) == \
        nbx.PARTIAL_TCGEN05                                   # verify window: 16 rows x 6 heads
    assert nbx.nbx_paged_decode_partial_kernel(nbx.NBX_BF16, nbx.NBX_BF16, 8, 32, 4, 128, 1000, 128) == \
        nbx.PARTIAL_TCGEN05                                   # exactly 64 query vectors
    simt = [(nbx.NBX_BF16, nbx.NBX_BF16, 1, 32, 8, 128, 1000, 16),     # single-row decode
            (nbx.NBX_BF16, nbx.NBX_BF16, 16, 24, 4, 256, 1000, 16),    # pages of 16 positions
            (nbx.NBX_F32, nbx.NBX_BF16, 16, 24, 4, 256, 1000, 64),     # fp32 queries
            (nbx.NBX_BF16, nbx.NBX_F32, 16, 24, 4, 256, 1000, 64),     # fp32 pool
            (nbx.NBX_BF16, nbx.NBX_BF16, 16, 24, 4, 64, 1000, 64),     # d = 64
            (nbx.NBX_BF16, nbx.NBX_BF16, 7, 36, 4, 128, 1000, 64),     # 63 query vectors
            (nbx.NBX_BF16, nbx.NBX_BF16, 16, 24, 4, 256, 2 ** 23, 64)]  # pool rows beyond 2^31 - 64
    for args in simt:
        assert nbx.nbx_paged_decode_partial_kernel(*args) == nbx.PARTIAL_SIMT, args
    # fp8 pool with a multi-row window: tensor cores on the codes (bf16 q only), no extra workspace
    assert nbx.nbx_paged_decode_partial_kernel(nbx.NBX_BF16, nbx.NBX_E4M3, 128, 24, 4, 256, 1000, 64) == \
        nbx.PARTIAL_TCGEN05_FP8
    assert nbx.nbx_paged_decode_partial_kernel(nbx.NBX_BF16, nbx.NBX_E4M3, 16, 24, 4, 128, 1000, 128) == \
        nbx.PARTIAL_TCGEN05_FP8
    assert nbx.nbx_paged_decode_partial_kernel(nbx.NBX_F32, nbx.NBX_E4M3, 128, 24, 4, 256, 1000, 64) == \
        nbx.PARTIAL_SIMT
    assert nbx.nbx_paged_decode_partial_kernel(nbx.NBX_BF16, nbx.NBX_E4M3, 8, 24, 4, 256, 1000, 64) == \
        nbx.PARTIAL_SIMT   # 48 query vectors
    base = nbx.nbx_paged_decode_workspace_bytes(1, 128, 24, 4, 256, 32768)
    for qd, pd in ((nbx.NBX_BF16, nbx.NBX_E4M3), (nbx.NBX_BF16, nbx.NBX_BF16), (nbx.NBX_F32, nbx.NBX_F32)):
        assert nbx.nbx_paged_decode_workspace_bytes_for(qd, pd, 1, 128, 24, 4, 256, 32768, 64) == base
    assert lib.nbx_paged_decode_partial_kernel(nbx.NBX_BF16, nbx.NBX_BF16, 16, 24, 5, 256, 10, 64) == -2
    assert lib.nbx_paged_decode_partial_kernel(nbx.NBX_BF16, nbx.NBX_BF16, 16, 24, 4, 256, 10, 40) == -4
    assert lib.nbx_paged_decode_partial_kernel(7, nbx.NBX_BF16, 16, 24, 4, 256, 10, 64) == -3


def test_fixed_shift_constants_match_the_printed_examples(lib):
    # maxdiffusion PR #477 prints C(N) and the gate for N = 4096 and N = 75,600 with Vmax = 256
    with open(os.path.join(ROOT, "tests", "golden", "fixed_m_constants.json")) as f:
        g = json.load(f)
    for c in g["cases"]:
        assert nbx.nbx_decode_fixed_shift_gate(c["n_keys"], g["v_max_bound"]) == (c["C"], c["gate"])
    # and the closed form at powers of two: C = 127 - log2 n - 8, gate = floor((C + 125) / 2)
    for lg in range(0, 20):
        C, gate = nbx.nbx_decode_fixed_shift_gate(1 << lg, 256.0)
        assert C == 119 - lg and gate == (C + 125) // 2
    with pytest.raises(nbx.NbxError):
        nbx.nbx_decode_fixed_shift_gate(0, 256.0)


def test_fixed_shift_entry_points_refuse_missing_bounds(lib):
    f = lib.nbx_paged_decode_attn_fixed_shift
    st = f(FAKE, 1, 2, 16, 8, 128, FAKE, FAKE, 1, 100, 2, 64, FAKE, 10, FAKE, 160, 0.1, 1.0, 1.0, FAKE, FAKE, 1 << 30,
           NULL, FAKE, NULL, NULL)
    assert st == -1
    st = lib.nbx_paged_decode_bounds(FAKE, 1, 2, 16, 8, 128, FAKE, FAKE, 1, 100, 2, 64, FAKE, 10, FAKE, 160, 1.0, 0.0,
                                     FAKE, FAKE, NULL, NULL)
    assert st == -8   # v_scale 0
