"""Lane-level models of the head_dim-128 value transform, checked on the CPU.

At head_dim 128 the value encoder and the value fetch give each row to two
lanes.  The lane of part p starts with the pairs P[j] = (element 64p + j,
element 64p + j + 32).  The transform is the unnormalised Sylvester-order
Walsh-Hadamard transform.  Strides 1..16 run across the pairs, stride 32 runs
inside each pair, and stride 64 crosses the two lanes.

The kernels' stride-64 stage moves half the data across lanes:
- the part-1 lane holds every pair swapped;
- both lanes send their second component in one shuffle;
- lane p ends with (element 32p + j, element 64 + 32p + j), the second
  negated when p = 1.

These models replay both forms in float32 with the kernels' operations and
operand order.  They check that the half-traffic form gives the plain form's
values bit for bit, in its own placement, and that both equal the
transform's definition.  CPU only.
"""
import numpy as np
import pytest

F = np.float32


def _stages_1_to_16(P):
    """Butterflies of strides 1..16 over 32 pairs, component-wise: (a, b) -> (a + b, a - b)."""
    for h in (1, 2, 4, 8, 16):
        for t in range(16):
            j = (t // h) * 2 * h + t % h
            a, b = P[j].copy(), P[j + h].copy()
            P[j], P[j + h] = a + b, a - b


def plain_two_lane(x):
    """The general form: stride 32 as (x + y, x - y), stride 64 by exchanging every value."""
    lanes = [np.stack([x[64 * p:64 * p + 32], x[64 * p + 32:64 * p + 64]], axis=1).astype(F) for p in (0, 1)]
    for P in lanes:
        _stages_1_to_16(P)
        a, b = P[:, 0].copy(), P[:, 1].copy()
        P[:, 0], P[:, 1] = a + b, a - b
    out = []
    for p in (0, 1):
        g = F(-1.0) if p else F(1.0)
        o = lanes[1 - p]
        out.append(lanes[p] * g + o)  # one rounding: g * P is exact
    y = np.empty(128, dtype=F)
    for p in (0, 1):
        y[64 * p:64 * p + 32] = out[p][:, 0]
        y[64 * p + 32:64 * p + 64] = out[p][:, 1]
    return y


def half_traffic_two_lane(x):
    """The head_dim-128 form: part-1 pairs swapped, one shuffle per pair, outputs re-owned."""
    lanes = []
    for p in (0, 1):
        lo, hi = x[64 * p:64 * p + 32], x[64 * p + 32:64 * p + 64]
        lanes.append(np.stack([hi, lo] if p else [lo, hi], axis=1).astype(F))
    for p, P in enumerate(lanes):
        _stages_1_to_16(P)
        s = F(-1.0) if p else F(1.0)
        xx, yy = P[:, 0].copy(), P[:, 1].copy()
        P[:, 0], P[:, 1] = s * xx + yy, (-s) * yy + xx  # fma(s, x, y), fma(-s, y, x): one rounding each
    sent = [P[:, 1].copy() for P in lanes]  # both lanes send their second component
    y = np.empty(128, dtype=F)
    for p, P in enumerate(lanes):
        a, o = P[:, 0], sent[1 - p]
        first, second = a + o, a - o
        y[32 * p:32 * p + 32] = first
        y[64 + 32 * p:96 + 32 * p] = -second if p else second  # the sign table undoes the negation
    return y


def sylvester(n):
    h = np.array([[1.0]])
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h


@pytest.mark.parametrize("seed", range(8))
def test_half_traffic_form_matches_plain_form_bit_for_bit(seed):
    rng = np.random.default_rng(seed)
    x = (rng.standard_t(5, 128) * np.exp(rng.normal(0, 1.5))).astype(F)
    a, b = plain_two_lane(x), half_traffic_two_lane(x)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("seed", range(4))
def test_both_forms_equal_the_transform(seed):
    rng = np.random.default_rng(100 + seed)
    x = rng.standard_normal(128).astype(F)
    want = sylvester(128) @ x.astype(np.float64)
    for y in (plain_two_lane(x), half_traffic_two_lane(x)):
        assert np.max(np.abs(y - want)) <= 1e-4 * np.max(np.abs(want))


def test_each_basis_vector_lands_in_its_column():
    """A dropped sign, a wrong owner lane or a transposed pair shows up as a wrong column."""
    H = sylvester(128)
    for k in range(128):
        e = np.zeros(128, dtype=F)
        e[k] = 1.0
        assert np.array_equal(half_traffic_two_lane(e), H[:, k].astype(F))


def test_groups_owned_by_each_lane():
    """After the transform lane p holds whole 32-groups p and 2 + p (its RMS and codes stay local)."""
    owned = {0: [], 1: []}
    for p in (0, 1):
        owned[p] = sorted({(32 * p + j) // 32 for j in range(32)} | {(64 + 32 * p + j) // 32 for j in range(32)})
    assert owned == {0: [0, 2], 1: [1, 3]}
