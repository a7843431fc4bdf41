"""Host logic of the graph-replayed block step: the cell ranges the
transition is sliced into."""
import pytest

from variable_length_batching_gb300.graph import slice_cuts


@pytest.mark.parametrize("P", [0, 1, 5, 157023, 956323])
@pytest.mark.parametrize("slices,growth", [(1, 2.0), (3, 1.0), (3, 2.0), (4, 3.0), (6, 1.5), (12, 2.0)])
def test_slice_cuts_cover_the_cells(P, slices, growth):
    c = slice_cuts(P, slices, growth)
    assert len(c) == slices + 1 and c[0] == 0 and c[-1] == P
    assert all(a <= b for a, b in zip(c, c[1:]))


def test_slice_cuts_sizes_follow_the_growth():
    # sevenths for three slices doubling: 1/7, 2/7, 4/7 of the cells
    assert slice_cuts(7000, 3, 2.0) == [0, 1000, 3000, 7000]
    assert slice_cuts(600, 6, 1.0) == [0, 100, 200, 300, 400, 500, 600]
    c = slice_cuts(10 ** 6, 4, 3.0)             # 1 : 3 : 9 : 27
    sizes = [b - a for a, b in zip(c, c[1:])]
    assert sizes == [25000, 75000, 225000, 675000]


def test_slice_cuts_rejects_bad_arguments():
    with pytest.raises(ValueError):
        slice_cuts(10, 0)
    with pytest.raises(ValueError):
        slice_cuts(10, 3, 0.0)
