"""GPU checks of the fixed-shift softmax (maxdiffusion PR #477, "fixed-m") on the tensor-core kernel.

The fixed shift changes how the weights are scaled, not what is computed: every output is checked
against the float64 oracle with the decode tolerance. Rows whose score bound passes the gate take the
fixed shift (the test checks from the bounds that they do); the page's adversarial input, which a
gate of W instead of floor(W / 2) would let through with part of the softmax mass flushed, must fall
back to the online max; a window whose P enters the product in f16 never takes it.
"""

import math

import numpy as np
import pytest
import torch

import bench
import oracle.paged as op
import paged_split_kv_append_gb300 as nbx
import workloads as wl
from tests import pins
from tests.test_gpu_parity import DEV, TOL

pytestmark = pytest.mark.gpu

LOG2E = 1.0 / math.log(2.0)


@pytest.fixture(scope="module", autouse=True)
def built():
    nbx.build()
    nbx.nbx_set_decode_grid_limit(0)
    yield


def _fixed_rows(case, q_norm, kv_max):
    """Which (b, r, h) rows pass the gate in every split, from the bounds and the split plan."""
    cfg = case.cfg
    qn = q_norm.cpu().numpy()
    kv = kv_max.cpu().numpy()
    ok = np.zeros((cfg.batch, cfg.rows, cfg.h_q), dtype=bool)
    for b in range(cfg.batch):
        bounds = op.split_bounds(int(case.lens[b]), cfg.page_tokens)
        n_max = max(hi - lo for lo, hi in zip(bounds, bounds[1:]))
        _, gate = nbx.nbx_decode_fixed_shift_gate(max(n_max, 1), 256.0)
        for h in range(cfg.h_q):
            hk = h // cfg.group
            U = qn[b, :, h] * kv[b, hk, 0] * case.scale * LOG2E
            ok[b, :, h] = (U <= gate) & (kv[b, hk, 1] <= 256.0)
    return ok


def _decode_both(case):
    sess = bench.session_for_case(case, DEV)
    online = sess.step().clone()
    q_norm, kv_max = nbx.nbx_paged_decode_bounds(sess.q, sess.k_pool, sess.v_pool, sess.block_table, sess.seq_lens,
                                                 sess.max_seq_len, sess.k_scale, sess.v_scale, status=sess.status)
    fixed = nbx.nbx_paged_decode_attn_fixed_shift(sess.q, sess.k_pool, sess.v_pool, sess.block_table, sess.seq_lens,
                                                  sess.max_seq_len, sess.scale, q_norm, kv_max, sess.k_scale,
                                                  sess.v_scale, status=sess.status)
    torch.cuda.synchronize()
    assert sess.status_bits() == 0
    return sess, online, fixed, q_norm, kv_max


def test_bounds_match_the_oracles_pools():
    case = wl.make_case("verify_small", device=DEV)
    sess, _, _, q_norm, kv_max = _decode_both(case)
    cfg = case.cfg
    kp, vp = pins.oracle_pools(case)
    qd = case.q.float().cpu().numpy().astype(np.float64)
    assert np.allclose(q_norm.cpu().numpy(), np.linalg.norm(qd, axis=-1), rtol=1e-5)
    for b in range(cfg.batch):
        L = int(case.lens[b])
        for hk in range(cfg.h_kv):
            K = op.read_sequence(kp, cfg.pool_dtype, case.k_scale, case.block_table[b], L, hk, cfg.page_tokens)
            V = op.read_sequence(vp, cfg.pool_dtype, case.v_scale, case.block_table[b], L, hk, cfg.page_tokens)
            assert abs(kv_max[b, hk, 0].item() - np.linalg.norm(K, axis=-1).max()) <= 1e-5 * np.linalg.norm(K, axis=-1).max()
            assert kv_max[b, hk, 1].item() == np.abs(V).max()


@pytest.mark.parametrize("name", ["verify_small"])
def test_fixed_shift_matches_the_oracle(name):
    case = wl.make_case(name, device=DEV)
    assert nbx.nbx_paged_decode_partial_kernel(nbx.NBX_BF16, nbx.NBX_BF16, case.cfg.rows, case.cfg.h_q, case.cfg.h_kv,
                                               case.cfg.d, 1, case.cfg.page_tokens) == nbx.PARTIAL_TCGEN05
    sess, online, fixed, q_norm, kv_max = _decode_both(case)
    assert _fixed_rows(case, q_norm, kv_max).all()      # every row takes the fixed shift
    assert not torch.equal(fixed, online)                # the weights were scaled another way
    want = pins.oracle_output(case)
    err = float(np.max(np.abs(fixed.cpu().numpy().astype(np.float64) - want)))
    assert err <= TOL["bf16"], err


def test_adversarial_bound_falls_back_to_the_online_max():
    # maxdiffusion PR #477, "Why the gate is floor(W/2) and not W": q = [235, 2], keys half [0, 1] and
    # half [0, -1], values +1 / -1 with the key's sign, logits +-2 in log2 units. The bound U = |q||k|
    # is about 235: inside W but not W/2. With a shift of ceil(U) - C the -2 logits would fall below
    # 2^-126 and flush, giving 1.0; the gate sends the rows to the online max, which gives
    # (4 - 1/4) / (4 + 1/4) = 15/17 for a row that sees as many keys of each sign.
    rows, h_q, h_kv, d, P, L = 16, 4, 1, 128, 64, 4096
    cfg = wl.Config("adv", 1, rows, h_q, h_kv, d, P, "bf16", "bf16", 7, ("fixed", (L,)))
    case = wl.make_case(cfg, device=DEV)
    case.q.zero_()
    case.q[..., 0] = 235.0
    case.q[..., 1] = 2.0
    sign = torch.where(torch.arange(L, device=DEV) % 2 == 0, 1.0, -1.0)
    case.k_raw.zero_()
    case.k_raw[:, 0, 1] = sign
    case.v_raw.zero_()
    case.v_raw[:, 0, :] = sign[:, None]
    case.scale = math.log(2.0)            # scale * q.k = +-2 ln 2: +-2 in log2 units
    sess, online, fixed, q_norm, kv_max = _decode_both(case)
    assert not _fixed_rows(case, q_norm, kv_max).any()   # the gate rejects every row
    assert torch.equal(fixed, online)
    want = pins.oracle_output(case)
    err = float(np.max(np.abs(fixed.cpu().numpy().astype(np.float64) - want)))
    assert err <= TOL["bf16"], err
    assert abs(float(fixed[0, rows - 1, 0, 0]) - 15.0 / 17.0) < 1e-3   # the last row sees 2048 of each sign


def test_f16_products_never_take_the_fixed_shift():
    # an fp8 window on tensor cores enters P in f16, which cannot hold 2^C: the online max throughout
    case = wl.make_case("prefill_small", device=DEV)
    sess, online, fixed, q_norm, kv_max = _decode_both(case)
    assert torch.equal(fixed, online)
