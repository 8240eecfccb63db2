"""GPU parity of plain decode (one query row, bf16 q and pools, d 128: the single-row configs) against
the float64 oracle, across GQA groups, page sizes and lengths around the kernel's 16-position tiles,
32-position stages and 512-position splits.

Same bars as the other decode tests: max |err| 2e-3 against the oracle, bit-identical under grid size
and page placement, pools starting as NaN so that any read past a sequence shows up.
"""

import numpy as np
import pytest
import torch

import bench
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


def rows_config(name, lens, h_q, h_kv, page, seed):
    cfg = wl.Config(name, len(lens[1]) if lens[0] == "fixed" else 6, 1, h_q, h_kv, 128, page, "bf16", "bf16", seed, lens)
    kind = nbx.nbx_paged_decode_partial_kernel(nbx.NBX_BF16, nbx.NBX_BF16, 1, h_q, h_kv, 128, 1000, page)
    assert kind == nbx.PARTIAL_SIMT, cfg
    return cfg


# GQA groups of 4, 1, 6 (a partial row block), 16 and 32; pages of 16 to 256 positions
@pytest.mark.parametrize("h_q,h_kv,page", [(32, 8, 16), (8, 8, 64), (24, 4, 32), (32, 2, 128), (32, 1, 16),
                                           (16, 1, 256)])
def test_head_layouts_and_page_sizes(h_q, h_kv, page):
    cfg = rows_config(f"rt_{h_q}_{h_kv}_{page}", ("uniform", 1, 3000), h_q, h_kv, page, 51)
    case = wl.make_case(cfg, device=DEV)
    sess, out = run_step(case)
    check_against_oracle(case, sess, out)
    for limit in (1, 3, 1000):
        _, o2 = run_step(case, grid_limit=limit)
        assert torch.equal(o2, out), f"grid limit {limit}"


# lengths at and around the 16-position tile, the 32-position stage, the 512-position split and
# longer splits; 0 (no unit, zero output)
EDGE = (0, 1, 15, 16, 17, 127, 128, 129, 255, 256, 257, 511, 512, 513, 767, 768, 769, 1023, 1024, 1025, 4097)


def test_edge_lengths_across_tiles():
    cfg = rows_config("rt_edges", ("fixed", EDGE), 32, 8, 16, 52)
    case = wl.make_case(cfg, device=DEV)
    sess, out = run_step(case)
    check_against_oracle(case, sess, out)
    assert np.all(out.cpu().numpy()[0] == 0.0)


def test_one_cta_runs_every_unit():
    # every unit-to-unit handover of the stage ring and the metadata slots on one CTA
    cfg = rows_config("rt_one", ("fixed", (1, 130, 64, 700, 257, 2049, 16, 385)), 24, 4, 16, 53)
    case = wl.make_case(cfg, device=DEV)
    _, ref = run_step(case)
    for limit in (1, 2, 5):
        sess, out = run_step(case, grid_limit=limit)
        assert sess.status_bits() == 0, f"grid limit {limit}: status {sess.status_bits():#x}"
        assert torch.equal(out, ref), f"grid limit {limit}"
    check_against_oracle(case, sess, out)


def ramp_case(rising: bool, seed: int):
    """One 2000-position sequence whose scores climb (or fall) steadily along the keys: with the keys
    along the query's direction, the running max of a rising ramp keeps growing by more than the lazy
    rescale's 2^8, so the accumulators are rescaled pass after pass; a falling ramp sets the max at
    the first keys and never rescales again."""
    cfg = rows_config("rt_ramp", ("fixed", (2000, 300)), 32, 8, 16, seed)
    case = wl.make_case(cfg, device=DEV)
    g = torch.Generator().manual_seed(seed)
    q = case.q.float().cpu()
    off = int(case.tok_offset[0])
    n = 2000
    steps = torch.arange(n, dtype=torch.float32) / n
    a = steps if rising else 1.0 - steps
    for h in range(cfg.h_kv):
        u = torch.randn(cfg.d, generator=g)
        u = u / u.norm()
        q[0, 0, h * cfg.group:(h + 1) * cfg.group] = 0.5 * q[0, 0, h * cfg.group:(h + 1) * cfg.group] + 3.0 * u
        base = case.k_raw[off:off + n, h].float().cpu()
        # q.k along u climbs by about 3 * 420 = 1260 over the sequence: 1260 / sqrt(128) * log2(e)
        # = 160 log2 units, about 10 per 128 positions
        k = 0.2 * base + 420.0 * a[:, None] * u[None, :]
        case.k_raw[off:off + n, h] = k.to(case.k_raw.dtype).to(case.k_raw.device)
    case.q.copy_(q.to(case.q.dtype).to(case.q.device))
    return case


@pytest.mark.parametrize("rising", [True, False])
def test_rescale_paths_match_the_oracle(rising):
    case = ramp_case(rising, 54)
    sess, out = run_step(case)
    check_against_oracle(case, sess, out)


def test_nan_key_and_value_reach_only_their_heads():
    cfg = rows_config("rt_nan", ("fixed", (1000, 300, 700)), 32, 8, 16, 55)
    case = wl.make_case(cfg, device=DEV)
    off = case.tok_offset
    case.k_raw[int(off[0]) + 700, 2, 9] = float("nan")     # sequence 0, KV head 2: a key
    case.v_raw[int(off[2]) + 5, 6, 100] = float("nan")     # sequence 2, KV head 6: a value
    sess, out = run_step(case)
    assert sess.status_bits() == 0
    o = out.cpu().numpy()
    G = cfg.group
    assert np.all(np.isnan(o[0, 0, 2 * G:3 * G]))
    assert np.all(np.isnan(o[2, 0, 6 * G:7 * G, 100])) and np.all(np.isfinite(o[2, 0, 6 * G:7 * G, :100]))
    want = pins.oracle_output(case)
    assert pins.nan_aware_error(o.astype(np.float64), want) <= 2e-3


def test_missing_page_sets_status_and_spares_other_sequences():
    cfg = rows_config("rt_bad", ("fixed", (900, 1300)), 32, 8, 16, 56)
    case = wl.make_case(cfg, device=DEV)
    sess = bench.session_for_case(case, DEV)
    bt = sess.block_table.clone()
    bt[1, 2] = -1
    bt[1, 40] = case.num_pages + 3
    sess.block_table = bt
    out = sess.step()
    torch.cuda.synchronize()
    assert sess.status_bits() & nbx.DEV_BAD_PAGE
    want = pins.oracle_output(case)
    got = out.cpu().numpy()
    assert np.max(np.abs(got[:1] - want[:1])) <= 2e-3
    assert np.all(np.isfinite(got[1]))     # the missing pages' positions are skipped
