"""The decode entry point for callers that cannot allocate device memory.

nbx_paged_decode_attn_noalloc runs the same decode as nbx_paged_decode_attn but keeps its
scratch (plan, work list, split partials) in a fixed array inside the library, so a caller that
cannot call cudaMalloc (an allocator callback, a plug-in without the host's allocator, a fixed
memory budget) only passes inputs and the output. This file is collected last on purpose.
"""

import ctypes

import numpy as np
import pytest
import torch

import bench
import paged_split_kv_append_gb300 as nbx
import workloads as wl
from tests import pins

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
TOL = {"f32": 2e-3, "bf16": 2e-3, "e4m3": 3e-2}   # fp32 output against the oracle: the decode parity tolerance
SCRATCH = 32 * 1024 * 1024


def _noalloc(lib):
    f = lib.nbx_paged_decode_attn_noalloc
    vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    f.argtypes = [vp, i32, i32, i32, i32, i32, vp, vp, i32, i32, i32, i32, vp, i32, vp, i32, f32, f32, f32, vp, vp,
                  vp]
    f.restype = i32
    return f


def _call(f, sess, out, status):
    q, kp = sess.q, sess.k_pool
    batch, rows, h_q, d = q.shape
    num_pages, h_kv, page_tokens, _ = kp.shape
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return f(ctypes.c_void_p(q.data_ptr()), nbx.dtype_code(q), batch, rows, h_q, d, ctypes.c_void_p(kp.data_ptr()),
             ctypes.c_void_p(sess.v_pool.data_ptr()), nbx.dtype_code(kp), num_pages, h_kv, page_tokens,
             ctypes.c_void_p(sess.block_table.data_ptr()), sess.block_table.shape[1],
             ctypes.c_void_p(sess.seq_lens.data_ptr()), sess.max_seq_len, sess.scale, sess.k_scale, sess.v_scale,
             ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(status.data_ptr()), stream)


@pytest.mark.parametrize("name,kernel", [("single_row", nbx.PARTIAL_SIMT), ("ragged_small", nbx.PARTIAL_SIMT),
                                         ("tiny", nbx.PARTIAL_SIMT),
                                         ("verify_small", nbx.PARTIAL_TCGEN05),
                                         ("prefill_small", nbx.PARTIAL_TCGEN05_FP8)])
def test_noalloc_decode_matches_the_workspace_decode_twice(name, kernel):
    # the same kernels with the same plan as the workspace entry point: the outputs are equal bit for bit
    nbx.build()
    lib = nbx.lib()
    f = _noalloc(lib)
    case = wl.make_case(name, device=DEV)
    cfg = case.cfg
    sess = bench.session_for_case(case, DEV)
    assert nbx.nbx_paged_decode_partial_kernel(nbx.dtype_code(sess.q), nbx.dtype_code(sess.k_pool), cfg.rows, cfg.h_q,
                                               cfg.h_kv, cfg.d, 1, cfg.page_tokens) == kernel
    ref = sess.step().clone()                  # the existing entry point, with its own workspace
    torch.cuda.synchronize()
    assert sess.status_bits() == 0
    # the fixed scratch holds what this call needs
    need = nbx.nbx_paged_decode_workspace_bytes_for(nbx.dtype_code(case.q), nbx.dtype_code(sess.k_pool), cfg.batch,
                                                    cfg.rows, cfg.h_q, cfg.h_kv, cfg.d, case.max_seq_len,
                                                    cfg.page_tokens)
    assert need <= SCRATCH
    for _ in range(2):                         # two calls in a row share the library's scratch
        out = torch.full_like(ref, float("nan"))
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        assert _call(f, sess, out, status) == 0
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(out, ref)
    if name != "single_row":                   # small enough for the oracle to compute every output
        want = pins.oracle_output(case)
        err = float(np.max(np.abs(out.cpu().numpy().astype(np.float64) - want)))
        assert err <= TOL[cfg.pool_dtype], err


def test_noalloc_rejects_sizes_beyond_its_scratch():
    nbx.build()
    f = _noalloc(nbx.lib())
    case = wl.make_case("single_row", device=DEV)
    sess = bench.session_for_case(case, DEV)
    # a bound of 131072 positions: 64 splits per row, more fp32 partials than the scratch holds
    sess.max_seq_len = 131072
    sess.block_table = torch.full((case.cfg.batch, 131072 // case.cfg.page_tokens), -1, dtype=torch.int32,
                                  device=DEV)
    need = nbx.nbx_paged_decode_workspace_bytes(case.cfg.batch, 1, case.cfg.h_q, case.cfg.h_kv, case.cfg.d, 131072)
    assert need > SCRATCH
    out = torch.zeros((case.cfg.batch, 1, case.cfg.h_q, case.cfg.d), device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    assert _call(f, sess, out, status) == -5   # NBX_ERR_WORKSPACE, nothing launched
    torch.cuda.synchronize()
    assert torch.all(out == 0) and int(status.item()) == 0
