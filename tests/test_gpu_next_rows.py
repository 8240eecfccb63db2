"""GPU checks of the calls beyond the core decode, through the C ABI.

- The graph-replayable decode step (nbxtensor/ops/paged_decode_attn.py, paged_kv_append_step_kernel
  and paged_lens_advance_kernel): positions come from the device lengths, which then advance, so
  one recorded step replays unchanged. Checked against the oracle (pools bit for bit, outputs within
  the decode tolerance) after the first step and after a graph-replayed second step, and bit for bit
  against the separate append + decode calls.
- The contiguous (non-paged) decode (nbxtensor/ops/attention_wrappers.py, _decode_attn_vec): a
  [batch, h_kv, capacity, d] cache read as one page per sequence. Checked against the oracle.
- Multi-row windows below the tensor-core threshold (rows x group < 64) on the SIMT kernel, with
  the rows-first unit order (TensorFold PR #1219). Checked against the oracle and across grid sizes.
"""

import numpy as np
import pytest
import torch

import bench
import oracle.paged as op
import paged_split_kv_append_gb300 as nbx
import workloads as wl
from tests import pins
from tests.test_gpu_parity import DEV, TOL, check_against_oracle, oracle_codes, pool_codes, run_step

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    nbx.build()
    nbx.nbx_set_decode_grid_limit(0)
    yield
    nbx.nbx_set_decode_grid_limit(0)


def _slots(block_table: torch.Tensor, P: int, b: int, pos: np.ndarray) -> np.ndarray:
    bt = block_table.cpu().numpy()
    return (bt[b, pos // P].astype(np.int64) * P + pos % P).astype(np.int32)


def _check_step_against_oracle(case, kp, vp, lens, q, k_pool, v_pool, out):
    """Pools bit for bit at every position the sequences hold, output within the tolerance of the
    oracle's decode over those pools."""
    cfg = case.cfg
    P = cfg.page_tokens
    pages = np.concatenate([case.block_table[b, np.arange(int(L)) // P] for b, L in enumerate(lens)])
    pos = np.concatenate([np.arange(int(L)) % P for L in lens])
    for gpu_pool, ora in ((k_pool, kp), (v_pool, vp)):
        got = pool_codes(gpu_pool, cfg.pool_dtype)[pages, :, pos, :]
        assert np.array_equal(got, oracle_codes(ora, cfg.pool_dtype)[pages, :, pos, :]), "step append not bit-exact"
    want = op.decode_attention(q.float().cpu().numpy(), kp, vp, cfg.pool_dtype, case.block_table,
                               np.asarray(lens), P, case.scale, case.k_scale, case.v_scale)
    err = float(np.max(np.abs(out.cpu().numpy().astype(np.float64) - want)))
    assert err <= TOL[cfg.pool_dtype], f"step: max abs error {err}"


# ------------------------------------------------------------------------------------ decode step
@pytest.mark.parametrize("rows,h_q,h_kv,d,P,pool", [(1, 8, 2, 128, 16, "bf16"), (4, 16, 4, 128, 32, "bf16"),
                                                    (16, 24, 4, 256, 64, "bf16"), (2, 8, 2, 64, 16, "e4m3")])
def test_decode_step_matches_append_then_decode_and_replays(rows, h_q, h_kv, d, P, pool):
    # lengths that leave room for a second step's rows in each sequence's last page
    lens = tuple(int(x) for x in (3 * P + rows, 5 * P - 2 * rows, 2 * P + 3, 9 * P + P // 2 - rows))
    cfg = wl.Config("step", len(lens), rows, h_q, h_kv, d, P, pool, "bf16", 41, ("fixed", lens))
    case = wl.make_case(cfg, device=DEV)
    assert np.all(case.lens >= rows)
    ref = bench.session_for_case(case, DEV)           # the pool holds len - rows positions
    pre_k, pre_v = ref.k_pool.clone(), ref.v_pool.clone()
    out_ref = ref.step().clone()                      # append at host slots, then decode
    B = cfg.batch
    new_k = ref.new_k.view(B, rows, h_kv, d)
    new_v = ref.new_v.view(B, rows, h_kv, d)
    lens_dev = (ref.seq_lens - rows).contiguous()
    k_pool, v_pool = pre_k.clone(), pre_v.clone()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    max_len = int(case.lens.max()) + rows             # room for the second step
    out = nbx.nbx_paged_decode_step(ref.q, new_k, new_v, k_pool, v_pool, ref.block_table, lens_dev, max_len,
                                    case.scale, case.k_scale, case.v_scale, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(lens_dev, ref.seq_lens)        # advanced by rows
    assert torch.equal(k_pool.view(torch.uint8), ref.k_pool.view(torch.uint8))
    assert torch.equal(v_pool.view(torch.uint8), ref.v_pool.view(torch.uint8))
    # the split plan is sized by max_seq_len, so compare with a reference sized the same way
    out_ref2 = nbx.nbx_paged_decode_attn(ref.q, ref.k_pool, ref.v_pool, ref.block_table, ref.seq_lens, max_len,
                                        case.scale, case.k_scale, case.v_scale)
    assert torch.equal(out, out_ref2)
    assert float((out - out_ref).abs().max()) <= TOL[pool]
    kp, vp = pins.oracle_pools(case)                  # the oracle appends the same tokens at the same slots
    _check_step_against_oracle(case, kp, vp, case.lens, ref.q, k_pool, v_pool, out)

    # a second step from a recorded graph: new keys at lens .. lens + rows - 1, lens advance again
    g = torch.Generator(device=DEV).manual_seed(7)
    new_k2 = torch.randn(new_k.shape, generator=g, device=DEV)
    new_v2 = torch.randn(new_v.shape, generator=g, device=DEV)
    nk, nv = new_k2.clone(), new_v2.clone()
    out2 = torch.empty_like(out)
    ws = torch.empty(max(nbx.nbx_paged_decode_workspace_bytes_for(nbx.NBX_BF16, nbx.dtype_code(k_pool), B, rows,
                                                                  h_q, h_kv, d, max_len, P), 256),
                     dtype=torch.uint8, device=DEV)
    stream = torch.cuda.Stream(device=DEV)
    graph = torch.cuda.CUDAGraph()
    lens_graph = lens_dev.clone()
    with torch.cuda.graph(graph, stream=stream):
        nbx.nbx_paged_decode_step(ref.q, nk, nv, k_pool, v_pool, ref.block_table, lens_graph, max_len, case.scale,
                                  case.k_scale, case.v_scale, out=out2, workspace=ws, status=status, stream=stream)
    lens_graph.copy_(lens_dev)            # capture does not run the kernels: start from the step-1 lengths
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(lens_graph, ref.seq_lens + rows)
    # the same second step through the separate calls
    slots = np.concatenate([_slots(ref.block_table, P, b, np.arange(int(case.lens[b]), int(case.lens[b]) + rows))
                            for b in range(B)])
    nbx.nbx_paged_kv_append(new_k2.view(B * rows, h_kv, d), new_v2.view(B * rows, h_kv, d), ref.k_pool,
                            ref.v_pool, torch.from_numpy(slots).to(DEV), case.k_scale, case.v_scale)
    lens2 = (ref.seq_lens + rows).contiguous()
    want = nbx.nbx_paged_decode_attn(ref.q, ref.k_pool, ref.v_pool, ref.block_table, lens2, max_len, case.scale,
                                     case.k_scale, case.v_scale)
    torch.cuda.synchronize()
    assert torch.equal(k_pool.view(torch.uint8), ref.k_pool.view(torch.uint8))
    assert torch.equal(out2, want)
    # and the oracle: step 2's own new tokens appended at the slots after step 1's lengths
    slots_np = slots.astype(np.int32)
    op.append(kp, new_k2.view(B * rows, h_kv, d).cpu().numpy(), slots_np, P, pool, case.k_scale)
    op.append(vp, new_v2.view(B * rows, h_kv, d).cpu().numpy(), slots_np, P, pool, case.v_scale)
    _check_step_against_oracle(case, kp, vp, case.lens + rows, ref.q, k_pool, v_pool, out2)


def test_decode_step_refuses_positions_past_the_bound():
    cfg = wl.Config("step_bad", 2, 2, 4, 2, 64, 16, "bf16", "bf16", 42, ("fixed", (40, 60)))
    case = wl.make_case(cfg, device=DEV)
    sess = bench.session_for_case(case, DEV)
    lens = (sess.seq_lens - 2).contiguous()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    new = torch.zeros((2, 2, 2, 64), device=DEV)
    # max_seq_len 50: sequence 1 would reach 60, so its new positions are refused and flagged
    nbx.nbx_paged_decode_step(sess.q, new, new, sess.k_pool, sess.v_pool, sess.block_table, lens, 50, case.scale,
                              status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & 0x4
    assert lens.tolist() == [40, 60]


# ------------------------------------------------------------------------------- contiguous cache
@pytest.mark.parametrize("name,capacity_pad", [("single_row_small", 0), ("single_row_small", 1000),
                                               ("verify_small", 64), ("prefill_small", 0)])
def test_contiguous_cache_matches_the_oracle(name, capacity_pad):
    case = wl.make_case(name, device=DEV)
    cfg = case.cfg
    sess, _ = run_step(case)                          # the pool now holds every position
    P = cfg.page_tokens
    align = 64 if cfg.rows * (cfg.h_q // cfg.h_kv) >= 64 else 16
    cap = -(-(int(case.lens.max()) + capacity_pad) // align) * align
    B, H, d = cfg.batch, cfg.h_kv, cfg.d
    kc = torch.zeros((B, H, cap, d), dtype=sess.k_pool.dtype, device=DEV)
    vc = torch.zeros_like(kc)
    bt = sess.block_table.long()
    for b in range(B):
        L = int(case.lens[b])
        j = torch.arange(L, device=DEV)
        pg = bt[b, j // P]
        kc[b, :, :L] = sess.k_pool[pg, :, j % P].permute(1, 0, 2)
        vc[b, :, :L] = sess.v_pool[pg, :, j % P].permute(1, 0, 2)
    if cfg.pool_dtype == "f32":
        kc[:, :, int(case.lens.max()):] = float("nan")   # positions no sequence holds stay unread
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = nbx.nbx_decode_attn_contiguous(sess.q, kc, vc, sess.seq_lens, int(case.lens.max()), case.scale,
                                         case.k_scale, case.v_scale, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = pins.oracle_output(case)
    err = float(np.max(np.abs(out.cpu().numpy().astype(np.float64) - ref)))
    assert err <= TOL[cfg.pool_dtype], f"{name}: max abs error {err}"


# -------------------------------------------------------------------- multi-row windows on SIMT
@pytest.mark.parametrize("rows,h_q,h_kv,d,P", [(4, 16, 4, 128, 16), (8, 24, 4, 256, 64), (3, 12, 4, 64, 32)])
def test_multi_row_window_below_the_tensor_core_threshold(rows, h_q, h_kv, d, P):
    assert rows * (h_q // h_kv) < 64
    assert nbx.nbx_paged_decode_partial_kernel(nbx.NBX_BF16, nbx.NBX_BF16, rows, h_q, h_kv, d, 1, P) == \
        nbx.PARTIAL_SIMT
    cfg = wl.Config("mr_simt", 5, rows, h_q, h_kv, d, P, "bf16", "bf16", 43, ("uniform", 300, 2500))
    case = wl.make_case(cfg, device=DEV)
    sess, out = run_step(case)
    check_against_oracle(case, sess, out)
    for limit in (1, 7, 1000):
        _, o2 = run_step(case, grid_limit=limit)
        assert torch.equal(o2, out), f"grid limit {limit}"


@pytest.mark.parametrize("d,pool", [(128, "bf16"), (64, "bf16"), (256, "bf16"), (128, "e4m3"), (128, "f32")])
def test_nan_past_a_rows_causal_limit_stays_out_of_that_row(d, pool):
    # A NaN value at the window's last position (the last row's own new token) is seen only by the
    # last row: the earlier rows of the window must match the oracle, which never reads past a row's
    # causal limit. A NaN key reaches exactly the rows that see it, including rows whose later
    # positions in the same split are masked (the NaN must survive those).
    rows, h_q, h_kv, P = 4, 16, 4, 16
    code = {"f32": nbx.NBX_F32, "bf16": nbx.NBX_BF16, "e4m3": nbx.NBX_E4M3}[pool]
    assert nbx.nbx_paged_decode_partial_kernel(nbx.NBX_BF16, code, rows, h_q, h_kv, d, 1, P) == nbx.PARTIAL_SIMT
    cfg = wl.Config("mr_nan", 4, rows, h_q, h_kv, d, P, pool, "bf16", 44, ("fixed", (100, 37, 256, 300)))
    case = wl.make_case(cfg, device=DEV)
    off = case.tok_offset
    case.v_raw[int(off[0]) + 99, 1, 5] = float("nan")        # sequence 0, last position: row 3 only
    case.v_raw[int(off[2]) + 254, 3, 0] = float("nan")       # sequence 2, next to last: rows 2 and 3
    case.k_raw[int(off[3]) + 298, 2, 7] = float("nan")       # sequence 3, a key rows 2 and 3 see
    case.k_raw[int(off[3]) + 170, 0, 3] = float("nan")       # sequence 3, early in its second split
    sess, out = run_step(case)
    assert sess.status_bits() == 0
    want = pins.oracle_output(case)
    got = out.cpu().numpy().astype(np.float64)
    assert np.isnan(want).any()
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    err = float(np.max(np.abs(got[ok] - want[ok])))
    assert err <= TOL[pool], err
