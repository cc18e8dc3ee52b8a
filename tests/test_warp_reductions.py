"""The warp reductions of the final-aggregation kernels (fullring.cu), emulated on the CPU with
an exact model of __shfl_xor_sync over 32 lanes: which lane ends with which warp total.

- warp_reduce_scatter (the slot-holding ring): 32 values per lane; after five butterfly steps
  ps[0] of lane L is the warp's total of value L.
- the pairwise reduce-scatter of the register-held kernel: four values per lane (square sum and
  query product of sources j0 and j0 + 1); lane bit 4 picks the source, lane bit 3 the sum, and
  the lanes 0, 8, 16, 24 store values 0, 1, 2, 3 at 2 j0 + lane / 8.

Integer-valued inputs make every sum exact, so the checks are equalities."""
import numpy as np
import pytest

LANES = np.arange(32)


def shfl_xor(vals, mask):
    """__shfl_xor_sync: lane L receives the value of lane L ^ mask."""
    return vals[LANES ^ mask]


def warp_reduce_scatter(ps):
    """ps: [32 lanes, 32 values]; returns ps[:, 0] after the kernel's butterfly."""
    ps = ps.copy()
    o = 16
    while o >= 1:
        upper = (LANES & o) != 0
        for i in range(o):
            send = np.where(upper, ps[:, i], ps[:, i + o])
            keep = np.where(upper, ps[:, i + o], ps[:, i])
            ps[:, i] = keep + shfl_xor(send, o)
        o >>= 1
    return ps[:, 0]


def pair_reduce_scatter(v4):
    """v4: [32 lanes, 4 values]; returns the value each lane holds after the kernel's steps."""
    up16 = (LANES & 16) != 0
    up8 = (LANES & 8) != 0
    k0 = np.where(up16, v4[:, 2], v4[:, 0]) + shfl_xor(np.where(up16, v4[:, 0], v4[:, 2]), 16)
    k1 = np.where(up16, v4[:, 3], v4[:, 1]) + shfl_xor(np.where(up16, v4[:, 1], v4[:, 3]), 16)
    t = np.where(up8, k1, k0) + shfl_xor(np.where(up8, k0, k1), 8)
    for m in (4, 2, 1):
        t = t + shfl_xor(t, m)
    return t


@pytest.mark.parametrize("seed", range(5))
def test_reduce_scatter_gives_lane_L_the_total_of_value_L(seed):
    rng = np.random.default_rng(seed)
    ps = rng.integers(-1000, 1000, size=(32, 32)).astype(np.float64)
    got = warp_reduce_scatter(ps)
    np.testing.assert_array_equal(got, ps.sum(axis=0))


@pytest.mark.parametrize("seed", range(5))
def test_pair_reduce_scatter_lane_map(seed):
    rng = np.random.default_rng(seed)
    v4 = rng.integers(-1000, 1000, size=(32, 4)).astype(np.float64)
    t = pair_reduce_scatter(v4)
    total = v4.sum(axis=0)
    for lane in range(32):
        assert t[lane] == total[((lane >> 4) & 1) * 2 + ((lane >> 3) & 1)], lane
    # the storing lanes (lane % 8 == 0) write value lane / 8 of the pair
    pw = np.full(32, np.nan)
    for j0 in (0, 2, 4, 6, 8):
        for lane in range(0, 32, 8):
            pw[2 * j0 + (lane >> 3)] = t[lane] + 100 * j0
    for j0 in (0, 2, 4, 6, 8):
        np.testing.assert_array_equal(pw[2 * j0:2 * j0 + 4], total + 100 * j0)


def test_pair_layout_matches_the_statistics_read():
    """The statistics read value 2j (square sum) and 2j + 1 (query product) of source j; the pair
    (j0, j0 + 1) stores (ss_j0, dot_j0, ss_j0+1, dot_j0+1) at 2 j0 .. 2 j0 + 3."""
    n = 10
    ss = np.arange(n) * 10.0 + 1
    dot = np.arange(n) * 10.0 + 2
    pw = np.zeros(32)
    for j0 in range(0, n, 2):
        v4 = np.zeros((32, 4))
        v4[0] = [ss[j0], dot[j0], ss[j0 + 1] if j0 + 1 < n else 0, dot[j0 + 1] if j0 + 1 < n else 0]
        t = pair_reduce_scatter(v4)
        for lane in range(0, 32, 8):
            pw[2 * j0 + (lane >> 3)] = t[lane]
    for j in range(n):
        assert pw[2 * j] == ss[j] and pw[2 * j + 1] == dot[j]
