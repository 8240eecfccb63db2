"""GPU parity: the CUDA path through the C ABI against the float64 oracle.

Bars (numerical contract): the append is bit-exact; the decode output (fp32) is within
max |err| 2e-3 of the oracle for fp32/bf16 pools and 3e-2 for fp8-e4m3 pools; the output
is bit-identical under a relabelling of physical pages, under any grid size and under a
reordering of the batch. Pools start filled with NaN, so a read of any position a
sequence does not hold would poison the output.
"""

import numpy as np
import pytest
import torch

import bench
import oracle.formats as fm
import oracle.paged as op
import paged_split_kv_append_gb300 as nbx
import workloads as wl
from tests import pins

pytestmark = pytest.mark.gpu

TOL = {"f32": 2e-3, "bf16": 2e-3, "e4m3": 3e-2}
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    nbx.build()
    nbx.nbx_set_decode_grid_limit(0)
    yield
    nbx.nbx_set_decode_grid_limit(0)


def pool_codes(t: torch.Tensor, dtype: str) -> np.ndarray:
    a = t.cpu()
    if dtype == "f32":
        return a.numpy().view(np.uint32)
    if dtype == "bf16":
        return a.view(torch.int16).numpy().view(np.uint16)
    return a.numpy().view(np.uint8)


def oracle_codes(pool: np.ndarray, dtype: str) -> np.ndarray:
    return pool.view(np.uint32) if dtype == "f32" else pool


def held_positions(case):
    P = case.cfg.page_tokens
    pages, pos = [], []
    for b in range(case.cfg.batch):
        j = np.arange(int(case.lens[b]))
        pages.append(case.block_table[b, j // P])
        pos.append(j % P)
    return np.concatenate(pages).astype(np.int64), np.concatenate(pos).astype(np.int64)


def run_step(case, grid_limit=0):
    nbx.nbx_set_decode_grid_limit(grid_limit)
    sess = bench.session_for_case(case, DEV)
    out = sess.step().clone()
    torch.cuda.synchronize()
    nbx.nbx_set_decode_grid_limit(0)
    return sess, out


def check_against_oracle(case, sess, out):
    cfg = case.cfg
    kp, vp = pins.oracle_pools(case)
    pg, ps = held_positions(case)
    for gpu_pool, ora in ((sess.k_pool, kp), (sess.v_pool, vp)):
        got = pool_codes(gpu_pool, cfg.pool_dtype)[pg, :, ps, :]
        want = oracle_codes(ora, cfg.pool_dtype)[pg, :, ps, :]
        assert np.array_equal(got, want), "append is not bit-exact"
    ref = pins.oracle_output(case, (kp, vp))
    got = out.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got))
    err = float(np.max(np.abs(got - ref)))
    assert err <= TOL[cfg.pool_dtype], f"{cfg.name}: max abs error {err}"
    assert sess.status_bits() == 0
    return err


@pytest.mark.parametrize("name", ["tiny", "single_row_small", "verify_small", "prefill_small", "ragged_small"])
def test_decode_matches_oracle(name):
    case = wl.make_case(name, device=DEV)
    sess, out = run_step(case)
    check_against_oracle(case, sess, out)


@pytest.mark.parametrize("lens", [[0, 1, 2, 15, 16, 17], [255, 256, 257, 4095, 4096, 4097], [16129, 1, 16385]])
def test_decode_edge_lengths(lens):
    case = wl.make_case("single_row_small", device=DEV, lens=lens)
    sess, out = run_step(case)
    check_against_oracle(case, sess, out)
    assert np.all(out.cpu().numpy()[np.array(lens) == 0] == 0.0)


@pytest.mark.parametrize("batch,hi", [(100, 900), (2100, 40)])
def test_decode_plan_paths_by_batch_size(batch, hi):
    # up to 2048 sequences are planned by the block-wide sort, more by the serial path; lengths of
    # 0 cover each path's empty sequences (output rows written as 0)
    cfg = wl.Config("plan_b%d" % batch, batch, 1, 4, 2, 64, 16, "bf16", "bf16", 31, ("uniform", 0, hi))
    lens = np.random.default_rng(batch).integers(0, hi + 1, batch)
    lens[::7] = 0
    case = wl.make_case(cfg, device=DEV, lens=[int(x) for x in lens])
    sess, out = run_step(case)
    check_against_oracle(case, sess, out)
    assert np.all(out.cpu().numpy()[case.lens == 0] == 0.0)


def test_decode_multi_row_short_sequences():
    # rows > length (some rows see no key), lengths ending mid-page, GQA group 3, fp32 queries
    cfg = wl.Config("mr", 5, 5, 6, 2, 64, 16, "bf16", "f32", 21, ("fixed", (3, 17, 1, 0, 40)))
    case = wl.make_case(cfg, device=DEV)
    sess, out = run_step(case)
    check_against_oracle(case, sess, out)


@pytest.mark.parametrize("pool_dtype,q_dtype,d", [("f32", "bf16", 128), ("bf16", "f32", 256), ("e4m3", "f32", 64),
                                                  ("e4m3", "bf16", 128), ("f32", "f32", 256), ("bf16", "bf16", 64)])
def test_decode_dtype_and_head_dim_grid(pool_dtype, q_dtype, d):
    cfg = wl.Config("grid", 3, 2, 8, 2, d, 32, pool_dtype, q_dtype, 22, ("uniform", 1, 900))
    case = wl.make_case(cfg, device=DEV)
    sess, out = run_step(case)
    check_against_oracle(case, sess, out)


def test_page_permutation_is_bit_exact():
    case = wl.make_case("ragged_small", device=DEV)
    _, out_a = run_step(case)
    _, bt2 = wl.permute_pages(case, seed=9)
    case2 = wl.Case(**{**case.__dict__, "block_table": bt2})
    _, out_b = run_step(case2)
    assert torch.equal(out_a, out_b)


@pytest.mark.parametrize("name", ["single_row_small", "verify_small"])
def test_grid_size_and_order_are_bit_exact(name):
    case = wl.make_case(name, device=DEV)
    _, ref = run_step(case)
    for limit in (1, 3, 37, 1000):
        _, out = run_step(case, grid_limit=limit)
        assert torch.equal(out, ref), f"grid limit {limit}"
    # reversed batch: every sequence's work runs at another place in the list
    perm = np.arange(case.cfg.batch)[::-1].copy()
    tok = [case.k_raw[int(case.tok_offset[b]):int(case.tok_offset[b + 1])] for b in perm]
    tokv = [case.v_raw[int(case.tok_offset[b]):int(case.tok_offset[b + 1])] for b in perm]
    off = np.zeros(case.cfg.batch + 1, dtype=np.int64)
    off[1:] = np.cumsum(case.lens[perm].astype(np.int64))
    case_r = wl.Case(**{**case.__dict__, "lens": case.lens[perm].copy(), "block_table": case.block_table[perm].copy(),
                        "tok_offset": off, "k_raw": torch.cat(tok), "v_raw": torch.cat(tokv), "q": case.q[perm.tolist()],
                        "n_new": case.n_new[perm].copy()})
    _, out_r = run_step(case_r)
    assert torch.equal(out_r, ref[perm.tolist()])


def test_repeated_calls_are_bit_identical():
    case = wl.make_case("verify_small", device=DEV)
    sess, out = run_step(case)
    for _ in range(3):
        again = sess.decode().clone()
        assert torch.equal(again, out)


def test_nan_key_reaches_the_output():
    # a NaN key in one split of a multi-split sequence: the merge skips only empty splits
    case = wl.make_case("single_row_small", device=DEV, lens=[1000, 300])
    case.k_raw[int(case.tok_offset[0]) + 700, 0, 5] = float("nan")
    sess, out = run_step(case)
    o = out.cpu().numpy()
    G = case.cfg.group
    assert np.all(np.isnan(o[0, 0, :G]))           # query heads of KV head 0
    assert np.all(np.isfinite(o[0, 0, G:])) and np.all(np.isfinite(o[1]))
    assert pins.nan_aware_error(o.astype(np.float64), pins.oracle_output(case)) <= TOL["bf16"]


def test_split_of_only_nan_keys_reaches_the_output():
    # every key of the second split is NaN (600 positions: two splits of 304 and 296 positions): its
    # running max is NaN, and the merge keeps it
    case = wl.make_case("single_row_small", device=DEV, lens=[600, 40])
    lo = int(case.tok_offset[0])
    case.k_raw[lo + 304:lo + 600, 1, :] = float("nan")
    sess, out = run_step(case)
    o = out.cpu().numpy()
    G = case.cfg.group
    assert np.all(np.isnan(o[0, 0, G:2 * G]))
    assert np.all(np.isfinite(o[0, 0, :G])) and np.all(np.isfinite(o[1]))
    assert pins.nan_aware_error(o.astype(np.float64), pins.oracle_output(case)) <= TOL["bf16"]


def test_a_wait_that_runs_out_sets_the_timeout_bit_and_returns():
    # every consumer warp's first wait (for its unit's queries) is bounded at 20 us while the producer
    # warps are held back 20 ms: the waits run out, the kernel records NBX_DEV_TIMEOUT, lets its copies
    # in flight land and returns. The call completes and the next call is correct.
    case = wl.make_case("single_row_small", device=DEV)
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


def test_bad_page_id_sets_status_and_skips():
    case = wl.make_case("single_row_small", device=DEV, lens=[100, 600])
    sess = bench.session_for_case(case, DEV)
    bt = sess.block_table.clone()
    bt[1, 3] = -1
    bt[1, 5] = case.num_pages + 7
    sess.block_table = bt
    out = sess.step()
    torch.cuda.synchronize()
    assert sess.status_bits() & nbx.DEV_BAD_PAGE
    kp, vp = pins.oracle_pools(case)
    ref = op.decode_attention(case.q.float().cpu().numpy()[:1], kp, vp, "bf16", case.block_table[:1], case.lens[:1],
                              16, case.scale)
    assert np.max(np.abs(out.cpu().numpy()[:1] - ref)) <= 2e-3   # the other sequence is untouched


def test_bad_length_sets_status():
    case = wl.make_case("single_row_small", device=DEV, lens=[100, 200])
    sess = bench.session_for_case(case, DEV)
    sess.seq_lens = torch.tensor([100, 10_000], dtype=torch.int32, device=DEV)
    out = sess.step()
    torch.cuda.synchronize()
    assert sess.status_bits() & nbx.DEV_BAD_LEN
    assert torch.all(out[1] == 0)


def test_append_bit_exact_with_edge_values():
    rng = np.random.default_rng(3)
    n, h, d, P = 40, 2, 64, 16
    x = (rng.standard_normal((n, h, d)) * 2.0 ** rng.integers(-14, 10, (n, h, d))).astype(np.float32)
    grid = np.unique(fm.e4m3_decode(np.arange(256, dtype=np.uint8)))
    grid = grid[np.isfinite(grid)]
    mids = ((grid[:-1] + grid[1:]) / 2).astype(np.float32)
    flat = x.reshape(-1)
    flat[:mids.size] = mids
    flat[mids.size:mids.size + 8] = [448.0, 464.0, 1e9, -1e9, np.inf, -np.inf, 0.0, -0.0]
    slots = rng.permutation(8 * P)[:n].astype(np.int32)
    for new_dtype in ("f32", "bf16"):
        src = torch.from_numpy(x)
        if new_dtype == "bf16":
            src = src.to(torch.bfloat16)
            xin = src.float().numpy()
        else:
            xin = x
        for pool_dtype, scale in (("f32", 1.0), ("bf16", 1.0), ("e4m3", 1.0), ("e4m3", 0.37)):
            kpool = bench_pool(8, h, P, d, pool_dtype)
            vpool = bench_pool(8, h, P, d, pool_dtype)
            nbx.nbx_paged_kv_append(src.to(DEV), src.to(DEV), kpool, vpool, torch.from_numpy(slots).to(DEV),
                                    k_scale=scale, v_scale=scale)
            torch.cuda.synchronize()
            ora = op.new_pool(8, h, P, d, pool_dtype)
            op.append(ora, xin, slots, P, pool_dtype, scale)
            got = pool_codes(kpool, pool_dtype)[slots // P, :, slots % P, :]
            want = oracle_codes(ora, pool_dtype)[slots // P, :, slots % P, :]
            assert np.array_equal(got, want), (new_dtype, pool_dtype, scale)
            assert np.array_equal(pool_codes(vpool, pool_dtype), pool_codes(kpool, pool_dtype))


def test_append_nan_input_stays_nan():
    x = torch.full((2, 1, 16), float("nan"), device=DEV)
    for pool_dtype in ("f32", "bf16", "e4m3"):
        pool = bench_pool(1, 1, 16, 16, pool_dtype, fill_nan=False)
        nbx.nbx_paged_kv_append(x, x, pool, pool, torch.tensor([0, 5], dtype=torch.int32, device=DEV))
        torch.cuda.synchronize()
        codes = pool_codes(pool, pool_dtype)[0, 0, [0, 5]]
        vals = fm.decode(codes if pool_dtype != "f32" else codes.view(np.float32), pool_dtype)
        assert np.all(np.isnan(vals))


def test_append_bad_slot_sets_status():
    x = torch.ones((3, 1, 16), device=DEV)
    pool = bench_pool(2, 1, 16, 16, "bf16", fill_nan=False)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    nbx.nbx_paged_kv_append(x, x, pool, pool, torch.tensor([3, -1, 32], dtype=torch.int32, device=DEV),
                            status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & nbx.DEV_BAD_SLOT
    codes = pool_codes(pool, "bf16")
    assert np.all(codes[0, 0, 3] == 0x3F80) and np.sum(codes != 0) == 16


def test_merge_matches_oracle():
    case = wl.make_case("ragged_small", device="cpu", lens=[3000, 70, 9000])
    kp, vp = pins.oracle_pools(case)
    cfg = case.cfg
    _, parts = op.decode_attention_split(case.q.float().numpy(), kp, vp, cfg.pool_dtype, case.block_table, case.lens,
                                         cfg.page_tokens, case.scale)
    keys = sorted(parts)
    S = max(len(parts[k][0]) for k in keys)
    m = np.full((len(keys), S), -np.inf, dtype=np.float32)
    l = np.zeros((len(keys), S), dtype=np.float32)
    acc = np.zeros((len(keys), S, cfg.d), dtype=np.float32)
    for i, k in enumerate(keys):
        ms, ls, accs = parts[k]
        m[i, :len(ms)] = ms
        l[i, :len(ms)] = ls
        acc[i, :len(ms)] = accs
    out = nbx.nbx_paged_decode_merge(torch.from_numpy(acc).to(DEV), torch.from_numpy(m).to(DEV),
                                     torch.from_numpy(l).to(DEV))
    ref = np.stack([op.merge(m[i].astype(np.float64), l[i].astype(np.float64), acc[i].astype(np.float64))
                    for i in range(len(keys))])
    assert np.max(np.abs(out.cpu().numpy() - ref)) <= 1e-5
    # all splits dead -> 0
    out0 = nbx.nbx_paged_decode_merge(torch.zeros((1, 4, 8), device=DEV), torch.full((1, 4), -np.inf, device=DEV),
                                      torch.zeros((1, 4), device=DEV))
    assert torch.all(out0 == 0)


def bench_pool(num_pages, h, P, d, dtype, fill_nan=True):
    from paged_split_kv_append_gb300.session import new_pool
    return new_pool(num_pages, h, P, d, dtype, DEV, fill_nan)


# ------------------------------------------------------------------------------ full-size workloads
def sampled_oracle(case, samples):
    """Oracle outputs for the sampled (b, r, h), from its own pools holding the sampled sequences."""
    cfg = case.cfg
    kp = op.new_pool(case.num_pages, cfg.h_kv, cfg.page_tokens, cfg.d, cfg.pool_dtype)
    vp = op.new_pool(case.num_pages, cfg.h_kv, cfg.page_tokens, cfg.d, cfg.pool_dtype)
    for b in sorted({s[0] for s in samples}):
        L = int(case.lens[b])
        lo, hi = int(case.tok_offset[b]), int(case.tok_offset[b + 1])
        slots = wl.slots_for(case.block_table, cfg.page_tokens, b, np.arange(L, dtype=np.int64))
        op.append(kp, case.k_raw[lo:hi].cpu().numpy(), slots, cfg.page_tokens, cfg.pool_dtype, case.k_scale)
        op.append(vp, case.v_raw[lo:hi].cpu().numpy(), slots, cfg.page_tokens, cfg.pool_dtype, case.v_scale)
    ref = op.decode_attention(case.q.float().cpu().numpy(), kp, vp, cfg.pool_dtype, case.block_table, case.lens,
                              cfg.page_tokens, case.scale, case.k_scale, case.v_scale, heads=samples)
    return ref, kp, vp


@pytest.mark.parametrize("name", ["single_row", "verify", "prefill", "ragged"])
def test_full_size_workload_sampled(name):
    cfg = wl.CONFIGS[name]
    case = wl.make_case(cfg, device=DEV)
    sess, out = run_step(case)
    assert sess.status_bits() == 0
    o = out.cpu().numpy()
    assert np.all(np.isfinite(o))
    rng = np.random.default_rng(7)
    order = np.argsort(case.lens)
    bs = sorted({int(order[-1]), int(order[0]), int(order[len(order) // 2]), int(rng.integers(cfg.batch))})
    samples = [(b, r, h) for b in bs for r in sorted({0, cfg.rows - 1, int(rng.integers(cfg.rows))})
               for h in sorted({0, cfg.h_q - 1, int(rng.integers(cfg.h_q))})]
    ref, kp, vp = sampled_oracle(case, samples)
    err = max(abs(float(np.max(np.abs(o[b, r, h] - ref[b, r, h])))) for b, r, h in samples)
    assert err <= TOL[cfg.pool_dtype], f"{name}: max abs error {err}"
    # the append of the sampled sequences is bit-exact
    P = cfg.page_tokens
    gpu_k = pool_codes(sess.k_pool, cfg.pool_dtype)
    for b in bs:
        j = np.arange(int(case.lens[b]))
        pg, ps = case.block_table[b, j // P].astype(np.int64), j % P
        assert np.array_equal(gpu_k[pg, :, ps, :], oracle_codes(kp, cfg.pool_dtype)[pg, :, ps, :])
