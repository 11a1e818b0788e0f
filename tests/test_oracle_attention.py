"""The fp64 attention oracle against its pins (CPU only)."""

import math

import numpy as np
import pytest

import oracle
import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(oracle)


@pytest.mark.parametrize("seed", [10, 11, 12])
def test_brute_force_more_layouts(seed):
    pins.check_brute_force(oracle, seed=seed, B=3, L=17, H=1, D=2, n_ids=2, p_pad=0.4)


def test_every_valid_row_admits_itself():
    q, k, v, do, sid = pins.rand_case(20, B=3, L=50, H=2, D=4, n_ids=5, p_pad=0.3)
    _, LSE = oracle.attention_fwd(q, k, v, sid)
    valid = sid >= 0
    assert np.isfinite(LSE.transpose(0, 2, 1)[valid]).all()
    assert np.isneginf(LSE.transpose(0, 2, 1)[~valid]).all()


def test_default_scale_is_inverse_sqrt_d():
    q, k, v, do, sid = pins.rand_case(21, B=1, L=12, H=1, D=9)
    a, la = oracle.attention_fwd(q, k, v, sid)
    b, lb = oracle.attention_fwd(q, k, v, sid, scale=1 / 3.0)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(la, lb)


def test_head_subset_matches_full():
    q, k, v, do, sid = pins.rand_case(22, B=2, L=20, H=3, D=4)
    O, LSE = oracle.attention_fwd(q, k, v, sid)
    O1, L1 = oracle.attention_fwd(q, k, v, sid, heads=[2])
    np.testing.assert_array_equal(O[:, :, 2:3], O1)
    np.testing.assert_array_equal(LSE[:, 2:3], L1)
    g = oracle.attention_bwd(q, k, v, do, sid)
    g1 = oracle.attention_bwd(q, k, v, do, sid, heads=[2])
    for a, b in zip(g[:3], g1[:3]):
        np.testing.assert_allclose(a[:, :, 2:3], b, rtol=0, atol=1e-14)


def test_query_blocking_is_summation_order_only():
    q, k, v, do, sid = pins.rand_case(23, B=1, L=70, H=1, D=4, n_ids=2)
    a = oracle.attention_bwd(q, k, v, do, sid, block=512)
    b = oracle.attention_bwd(q, k, v, do, sid, block=7)
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, rtol=0, atol=1e-12)


def test_effective_pairs_brute_force():
    _, _, _, _, sid = pins.rand_case(24, B=3, L=30, n_ids=4)
    brute = sum(1 for b in range(3) for i in range(30) for j in range(30)
                if sid[b, i] >= 0 and sid[b, i] == sid[b, j])
    assert oracle.effective_pairs(sid) == brute


def test_bf16_inputs_are_upcast_exactly():
    torch = pytest.importorskip("torch")
    q, k, v, do, sid = pins.rand_case(25, B=1, L=16, H=2, D=8)
    tq, tk, tv = (torch.tensor(x).to(torch.bfloat16) for x in (q, k, v))
    O_t, _ = oracle.attention_fwd(tq, tk, tv, sid)
    O_n, _ = oracle.attention_fwd(*(t.to(torch.float64).numpy() for t in (tq, tk, tv)), sid)
    np.testing.assert_array_equal(O_t, O_n)
    assert math.isclose(float(tq.to(torch.float64)[0, 0, 0, 0]), float(tq[0, 0, 0, 0]))
