"""The GPU tests' log re-indexing (tests/gpu_helpers.linear_log) against the layout the
header documents: CTA tiles row-major over (M / 128) x (N / bn) per problem, problems in
order; cluster tile c sits at raster position (m, n), and the CTA of rank r covers row
block m * RM + r // RN and column block n * RN + r % RN.  No GPU: the log is synthesised
from that description and must come back as one owner and one claim per cluster tile."""
import pytest

from oracle import coverage as cv

pytest.importorskip("torch")
from tests.gpu_helpers import linear_log  # noqa: E402


@pytest.mark.parametrize("cl,rn", [(1, 1), (2, 1), (4, 1), (4, 2)])
@pytest.mark.parametrize("group_rows", [1, 3, 16])
def test_linear_log_recovers_cluster_tiles(cl, rn, group_rows):
    rm = cl // rn
    problems = [(5, 3), (0, 2), (7, 1)]            # (cluster-tile rows, cluster-tile columns)
    n_tiles = sum(mt * nt for mt, nt in problems) * cl
    owner = [-1] * n_tiles
    claims = [0] * n_tiles
    base = 0
    for mt, nt in problems:
        for c in range(mt * nt):
            m, n = cv.raster(c, mt, nt, group_rows)
            for r in range(cl):
                row, col = m * rm + r // rn, n * rn + r % rn
                pos = base * cl + row * (nt * rn) + col
                owner[pos] = 1000 + base + c          # the worker that ran cluster tile c
                claims[pos] = 1
        base += mt * nt
    assert -1 not in owner
    owner_lin, claims_lin = linear_log(owner, claims, [p[0] for p in problems], [p[1] for p in problems], cl,
                                       group_rows=group_rows, rn=rn)
    assert owner_lin == [1000 + i for i in range(len(owner_lin))]
    assert claims_lin == [1] * len(claims_lin)


def test_linear_log_rejects_split_cluster_owners():
    owner = [7, 7, 8, 7]      # one cluster tile of 4 CTAs whose CTAs logged different workers
    claims = [1, 1, 1, 1]
    with pytest.raises(AssertionError):
        linear_log(owner, claims, [1], 1, 4, rn=2)
