"""GPU parity of the tensor-core split partial (tcgen05) against the float64 oracle.

The decode runs this kernel when the query vectors of one KV head fill an MMA tile
(rows x group >= 64, bf16 q, bf16 or E4M3 pools, d 128 or 256, pages of a multiple of 64
positions): multi-row verify windows and prefill chunks. Same bars as the SIMT kernel: max |err|
2e-3 for bf16 pools and 3e-2 for E4M3 pools, bit-identical under page relabelling, grid size and
batch order; pools start as NaN.
"""

import numpy as np
import pytest
import torch

import bench
import oracle.paged as op
import paged_split_kv_append_gb300 as nbx
import workloads as wl
from tests import pins
from tests.test_gpu_parity import DEV, check_against_oracle, run_step

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    nbx.build()
    nbx.nbx_set_decode_grid_limit(0)
    yield
    nbx.nbx_set_decode_grid_limit(0)


def tc_config(name, batch, rows, h_q, h_kv, d, page, lens, seed):
    cfg = wl.Config(name, batch, rows, h_q, h_kv, d, page, "bf16", "bf16", seed, lens)
    kind = nbx.nbx_paged_decode_partial_kernel(nbx.NBX_BF16, nbx.NBX_BF16, rows, h_q, h_kv, d, 1000, page)
    assert kind == nbx.PARTIAL_TCGEN05, cfg
    return cfg


# lengths around the 64-position tile, the 256-position split grain and the page; 0 and
# lengths below the window (rows that see no key)
EDGE_LENS = (0, 1, 15, 16, 17, 63, 64, 65, 257, 511, 512, 513, 4097)


def test_verify_window_edge_lengths():
    cfg = tc_config("tc_edges", len(EDGE_LENS), 16, 24, 4, 256, 64, ("fixed", EDGE_LENS), 31)
    case = wl.make_case(cfg, device=DEV)
    sess, out = run_step(case)
    check_against_oracle(case, sess, out)
    o = out.cpu().numpy()
    assert np.all(o[0] == 0.0)                     # empty sequence
    assert np.all(o[1, :15] == 0.0)                # length 1: rows 0..14 see no key


def test_head_dim_128_with_exactly_one_half_tile():
    # 8 rows x group 8 = 64 query vectors: half of the 128-lane tile is padding
    cfg = tc_config("tc_d128", 4, 8, 32, 4, 128, 64, ("uniform", 1, 3000), 32)
    case = wl.make_case(cfg, device=DEV)
    sess, out = run_step(case)
    check_against_oracle(case, sess, out)


def test_several_query_tiles_per_head():
    # 32 rows x group 6 = 192 query vectors: two M tiles per (split, KV head), pages of 128
    cfg = tc_config("tc_mtiles", 2, 32, 24, 4, 256, 128, ("uniform", 20, 2000), 33)
    case = wl.make_case(cfg, device=DEV)
    sess, out = run_step(case)
    check_against_oracle(case, sess, out)


def test_page_permutation_is_bit_exact():
    case = wl.make_case("verify_small", device=DEV)
    _, out_a = run_step(case)
    _, bt2 = wl.permute_pages(case, seed=5)
    case2 = wl.Case(**{**case.__dict__, "block_table": bt2})
    _, out_b = run_step(case2)
    assert torch.equal(out_a, out_b)


def test_grid_limits_with_several_query_tiles_are_bit_exact():
    cfg = tc_config("tc_mtiles_grid", 2, 32, 24, 4, 256, 64, ("fixed", (1500, 700)), 34)
    case = wl.make_case(cfg, device=DEV)
    _, ref = run_step(case)
    for limit in (1, 5, 151, 4000):
        _, out = run_step(case, grid_limit=limit)
        assert torch.equal(out, ref), f"grid limit {limit}"


def test_nan_key_reaches_only_its_heads():
    case = wl.make_case("verify_small", device=DEV, lens=[1000, 300])
    case.k_raw[int(case.tok_offset[0]) + 700, 0, 9] = float("nan")
    _, out = run_step(case)
    o = out.cpu().numpy()
    G = case.cfg.group
    assert np.all(np.isnan(o[0, :, :G]))           # every row of sequence 0 sees position 700
    assert np.all(np.isfinite(o[0, :, G:])) and np.all(np.isfinite(o[1]))


def test_missing_page_sets_status_and_spares_other_sequences():
    case = wl.make_case("verify_small", device=DEV, lens=[900, 1300])
    sess = bench.session_for_case(case, DEV)
    bt = sess.block_table.clone()
    bt[1, 2] = -1
    bt[1, 4] = case.num_pages + 3
    sess.block_table = bt
    out = sess.step()
    torch.cuda.synchronize()
    assert sess.status_bits() & nbx.DEV_BAD_PAGE
    kp, vp = pins.oracle_pools(case)
    ref = op.decode_attention(case.q.float().cpu().numpy()[:1], kp, vp, "bf16", case.block_table[:1], case.lens[:1],
                              case.cfg.page_tokens, case.scale)
    assert np.max(np.abs(out.cpu().numpy()[:1] - ref)) <= 2e-3
    assert np.all(np.isfinite(out.cpu().numpy()[1]))   # the missing pages' positions are skipped


@pytest.mark.parametrize("d,h_q,h_kv,page", [(256, 24, 4, 64), (128, 32, 4, 64)])
def test_one_cta_runs_every_unit(d, h_q, h_kv, page):
    # many short units (1-4 tiles, 1-3 splits) queued on one CTA, then on a few: every unit-to-unit
    # handover of the shared-memory rings and TMEM, compared with the oracle and the default grid
    lens = (1, 17, 64, 65, 130, 200, 257, 700, 64, 129)
    cfg = tc_config(f"tc_seq_d{d}", len(lens), 16, h_q, h_kv, d, page, ("fixed", lens), 35)
    case = wl.make_case(cfg, device=DEV)
    _, ref = run_step(case)
    for limit in (1, 2, 7):
        sess, out = run_step(case, grid_limit=limit)
        assert sess.status_bits() == 0, f"grid limit {limit}: status {sess.status_bits():#x}"
        assert torch.equal(out, ref), f"grid limit {limit}"
    check_against_oracle(case, sess, out)


def fp8_config(name, lens, seed, rows=16, page=64, h_q=24, h_kv=4, d=256):
    cfg = wl.Config(name, len(lens), rows, h_q, h_kv, d, page, "e4m3", "bf16", seed, ("fixed", tuple(lens)))
    kind = nbx.nbx_paged_decode_partial_kernel(nbx.NBX_BF16, nbx.NBX_E4M3, rows, h_q, h_kv, d, 1000, page)
    assert kind == nbx.PARTIAL_TCGEN05_FP8
    return cfg


def test_fp8_pool_window_on_the_codes():
    # kind::f8f6f4 on the stored codes, Q and P as two E4M3 terms each: held to the fp8 bound
    cfg = fp8_config("tc_fp8", (1, 64, 100, 700, 1500), 36)
    case = wl.make_case(cfg, device=DEV)
    sess, out = run_step(case)
    check_against_oracle(case, sess, out)


@pytest.mark.parametrize("rows,h_q,h_kv,page", [(16, 32, 4, 128), (8, 64, 2, 64)])
def test_fp8_window_head_dim_128(rows, h_q, h_kv, page):
    # d = 128: one 128-code atom per K and V tile row (the d = 256 windows have two); a group of 8
    # (one full M tile of 16 rows) on 128-position pages, and a group of 32 (two tiles of 4 rows)
    cfg = fp8_config(f"tc_fp8_d128_{h_q}", (1, 63, 64, 65, 700, 2500), 44, rows=rows, page=page, h_q=h_q,
                     h_kv=h_kv, d=128)
    case = wl.make_case(cfg, device=DEV)
    sess, out = run_step(case)
    check_against_oracle(case, sess, out)
    _, o2 = run_step(case, grid_limit=3)
    assert torch.equal(o2, out)


@pytest.mark.parametrize("name", ["verify_small", "prefill_small"])
def test_a_tensor_core_wait_that_runs_out_sets_the_timeout_bit_and_returns(name):
    # The producer warps are held back 20 ms and every wait is bounded at 20 us: the MMA issuers'
    # and the softmax warps' waits run out, the kernel records NBX_DEV_TIMEOUT, lets the copies the
    # producers then issue land, waits for its MMAs, releases its TMEM and returns. The call
    # completes and the next call is correct (bf16 and fp8 pools).
    case = wl.make_case(name, device=DEV)
    sess = bench.session_for_case(case, DEV)
    torch.cuda.synchronize()
    try:
        nbx.nbx_set_decode_wait_test(20_000, 20_000_000)
        sess.step()
        torch.cuda.synchronize()
    finally:
        nbx.nbx_set_decode_wait_test(0, 0)
    assert sess.status_bits() & nbx.DEV_TIMEOUT
    sess.status.zero_()
    out = sess.decode().clone()
    torch.cuda.synchronize()
    check_against_oracle(case, sess, out)


def fp8_scored_case(name, lens, seed, score_log2):
    """An fp8 window whose query vectors are all one vector q0 (every row and head) and whose key j
    is t_j q0 / |q0|^2 in every KV head, t_j set so that the score of position j is score_log2(j)
    in log2 units (up to the E4M3 rounding of the keys): the score pattern is placed position by
    position."""
    cfg = fp8_config(name, lens, seed)
    case = wl.make_case(cfg, device=DEV)
    case.q[:] = case.q[0, 0, 0]
    q0 = case.q[0, 0, 0].float()
    for b in range(cfg.batch):
        off, n = int(case.tok_offset[b]), int(case.lens[b])
        t = torch.tensor([score_log2(b, j, n) for j in range(n)], dtype=torch.float32, device=q0.device)
        t = t / (case.scale * np.log2(np.e))
        case.k_raw[off:off + n] = (t[:, None] * q0 / (q0 @ q0))[:, None, :]
    return wl.Case(**{**case.__dict__, "k_scale": float(case.k_raw.abs().max()) / wl.E4M3_MAX,
                      "v_scale": float(case.v_raw.abs().max()) / wl.E4M3_MAX})


def test_fp8_attention_sink_with_heavy_tail():
    # One key 10 log2 units above 1,500 others at ~0: each of those weighs ~2^-10 of the sink, below
    # what one E4M3 term holds next to it, yet together they outweigh it. The running max moves
    # back down after the sink's tile so their weights keep their bits. The sink sits in the first
    # tile of sequence 0 and in the middle of sequence 1.
    def score(b, j, n):
        return 10.0 if j == (3 if b == 0 else n // 2) else 0.05 * np.sin(0.7 * j)
    case = fp8_scored_case("tc_fp8_sink", (1500, 1700), 41, score)
    sess, out = run_step(case)
    check_against_oracle(case, sess, out)
    # the tail matters: attending to the sink alone would be far off
    kp, vp = pins.oracle_pools(case)
    want = pins.oracle_output(case)
    off = int(case.tok_offset[0])
    v_sink = case.v_raw[off + 3].float().cpu().numpy()   # ~ the dequantised sink value row of each KV head
    assert np.max(np.abs(want[0, 0, 0] - v_sink[0])) > 0.2


def test_fp8_flat_tail_far_below_a_sink():
    # Every query vector is e_0 and key j is t_j e_0, so a score is t_j * scale exactly (the sink's
    # key is the pool's largest, code 448): a sink 13.415 log2 units above 5,999 zero-score keys.
    # With m 5 below the sink each tail weight is 2^-8.415 = 1.498 * 2^-9, which the E4M3 terms
    # round to 2^-8 (+33 %), the same way for every key. The tail holds a fifth of the weight and
    # its values are all +3 (the sink's -3). A window of 128 rows over 6,000 keys is cut into
    # splits of 1,024: an output that kept the sink split's tail weights would be off by ~0.1.
    # The floor budget moves m down after two tail tiles, after which the tail's weights keep
    # their bits (off by ~0.014).
    cfg = fp8_config("tc_fp8_flat", (6000,), 43, rows=128)
    case = wl.make_case(cfg, device=DEV)
    case.q.zero_()
    case.q[..., 0] = 1.0
    b_sink = 13.415 / (case.scale * np.log2(np.e))
    case.k_raw.zero_()
    case.v_raw.fill_(3.0)
    for b in range(cfg.batch):
        sink = int(case.tok_offset[b]) + 3
        case.k_raw[sink, :, 0] = b_sink
        case.v_raw[sink] = -3.0
    case = wl.Case(**{**case.__dict__, "k_scale": b_sink / wl.E4M3_MAX, "v_scale": 3.0 / wl.E4M3_MAX})
    sess, out = run_step(case)
    check_against_oracle(case, sess, out)


@pytest.mark.parametrize("slope", [-2.0, -40.0, 2.0])
def test_fp8_score_ramps(slope):
    # scores changing by `slope` log2 units per 64-position tile: falling ramps move the running max
    # down tile after tile until the gathered weight reaches its bound (-2: gently; -40: at once),
    # a rising one moves it up
    case = fp8_scored_case("tc_fp8_ramp", (1400, 900), 42, lambda b, j, n: slope * j / 64.0)
    sess, out = run_step(case)
    check_against_oracle(case, sess, out)


def test_fp8_grid_limits_are_bit_exact():
    cfg = fp8_config("tc_fp8_grid", (130, 1500, 64), 37, rows=32)
    case = wl.make_case(cfg, device=DEV)
    _, ref = run_step(case)
    for limit in (1, 3, 200):
        sess, out = run_step(case, grid_limit=limit)
        assert sess.status_bits() == 0
        assert torch.equal(out, ref), f"grid limit {limit}"


def test_fp8_missing_page_and_nan_code():
    cfg = fp8_config("tc_fp8_bad", (900, 1300), 38)
    case = wl.make_case(cfg, device=DEV)
    case.k_raw[int(case.tok_offset[0]) + 500, 2, 7] = float("nan")   # stored as the E4M3 NaN code
    sess = bench.session_for_case(case, DEV)
    bt = sess.block_table.clone()
    bt[1, 3] = -1
    sess.block_table = bt
    out = sess.step()
    torch.cuda.synchronize()
    assert sess.status_bits() & nbx.DEV_BAD_PAGE
    o = out.cpu().numpy()
    G = cfg.group
    assert np.all(np.isnan(o[0, :, 2 * G:3 * G]))          # every row of sequence 0 sees position 500
    assert np.all(np.isfinite(o[0, :, :2 * G])) and np.all(np.isfinite(o[1]))
    kp, vp = pins.oracle_pools(case)
    ref = op.decode_attention(case.q.float().cpu().numpy()[:1], kp, vp, "e4m3", case.block_table[:1], case.lens[:1],
                              cfg.page_tokens, case.scale, case.k_scale, case.v_scale)
    keep = np.isfinite(ref)
    assert np.max(np.abs(o[:1][keep] - ref[keep])) <= 3e-2


def test_nan_key_reaches_rows_whose_later_tiles_are_masked():
    # prefill window: 128 rows at 1372..1499 of a 1500-position sequence; the last split is
    # [1280, 1500). A NaN key at 1300 is seen by every row, and the rows before 1408 then meet
    # 64-position tiles they cannot see: the NaN must survive those tiles (the oracle gives NaN
    # for every row of that KV head) and stay out of the other heads.
    case = wl.make_case("prefill_small", device=DEV)
    case.k_raw[1300, 1, 9] = float("nan")
    sess = bench.session_for_case(case, DEV)
    assert nbx.nbx_paged_decode_partial_kernel(nbx.NBX_BF16, nbx.NBX_E4M3, 128, 24, 4, 256, 1, 64) == \
        nbx.PARTIAL_TCGEN05_FP8
    out = sess.step().clone()
    torch.cuda.synchronize()
    assert sess.status_bits() == 0
    want = pins.oracle_output(case)
    got = out.cpu().numpy().astype(np.float64)
    G = case.cfg.group
    assert np.all(np.isnan(want[0, :, G:2 * G]))
    assert pins.nan_aware_error(got, want) <= 3e-2


def test_several_whole_row_query_tiles_per_head():
    # 32 rows x group 8 = 256 query vectors: two M tiles of 16 whole rows each, so each tile's query
    # block is one tensor box (the second at row 16); compared with the oracle and across grid sizes
    cfg = tc_config("tc_whole_rows", 3, 32, 32, 4, 128, 64, ("uniform", 40, 3000), 39)
    case = wl.make_case(cfg, device=DEV)
    sess, out = run_step(case)
    check_against_oracle(case, sess, out)
    for limit in (1, 5):
        _, o2 = run_step(case, grid_limit=limit)
        assert torch.equal(o2, out), f"grid limit {limit}"


def test_fp8_window_partials_at_the_code_range_edge():
    # An fp8 window stores each split's partial as f16 acc / l. Make every head attend almost
    # entirely to one position whose value row holds the largest codes (+-448, the amax row that
    # sets the v scale): the partials then sit at the edge of the E4M3 range, and the output must
    # still match the oracle.
    cfg = fp8_config("tc_fp8_edge", (2000, 1500), 40)
    case = wl.make_case(cfg, device=DEV)
    G = cfg.group
    for b in range(cfg.batch):
        off = int(case.tok_offset[b])
        n = int(case.lens[b])
        for h in range(cfg.h_kv):
            pos = off + (37 * (h + 1) + 11 * b) % n
            qv = case.q[b, :, h * G:(h + 1) * G].float().mean(dim=(0, 1))
            case.k_raw[pos, h] = (8.0 * qv / qv.norm()).to(case.k_raw.dtype)
            case.v_raw[pos, h] = torch.where(torch.arange(cfg.d, device=case.v_raw.device) % 2 == 0, 6.0, -6.0).to(
                case.v_raw.dtype)
    # the per-tensor scales follow the raw values (amax / 448)
    case = wl.Case(**{**case.__dict__, "k_scale": float(case.k_raw.abs().max()) / wl.E4M3_MAX,
                      "v_scale": float(case.v_raw.abs().max()) / wl.E4M3_MAX})
    sess, out = run_step(case)
    err = check_against_oracle(case, sess, out)
    assert err <= 3e-2, err
